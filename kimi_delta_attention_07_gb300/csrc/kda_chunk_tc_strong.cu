// Strong-decay prep of the tensor-core chunk path: the (chunk, head) items
// that the main prep (kda_chunk_tc.cu) deferred because a key channel decays by
// more than its single chunk-wide exponential reference can carry (a
// log-decay span beyond 80 on either side of the chunk's middle token).  The
// model's lower-bounded gate at -5 (decays of up to -5 per token) sends about
// half of its chunks here.
//
// Same outputs as the main prep (the per-(chunk, head) record of the state
// scan), from the chunked form of the Ascend model file's _torch_chunk_kda,
// with the decay referenced per 16-token block instead:
//   * G is replaced in place by l_r = exp(G_r - G_{16 br}) (br = r's 16-row
//     block); rho_b = exp(G_{16b}), so exp(G_r) = l_r * rho_br.  Every
//     exponent here is <= 0.
//   * Causal scores A[r,j] and the interaction matrix L[r,j] come from ONE
//     M=128 x N=160 x K=128 MMA: the A operand is [q_hat l ; k_hat l] (row
//     r referenced to its own block start), the B operand stacks, for the
//     10 (row block br, column block b) pairs with br >= b, the 16 rows
//     k_hat_j * exp(G_{16br} - G_j), j in block b.  Row r of block br finds
//     its columns j < 16(br+1) side by side.  Off the block diagonal both
//     factors are <= 1, so the products are exact or negligibly small for any
//     decay; on the diagonal the column factor is at most exp(15 max|g|).
//     A block whose decay span exceeds 75 (per-token decays below about -5)
//     has its diagonal 16 x 16 scores recomputed from exact pairwise
//     exponentials after the MMA (KDA_WS_EXACT_DECAY).
//   * X = (I + beta L)^-1 blockwise in fp32: 16x16 diagonal blocks by
//     forward substitution (one column per lane), the rest as
//     (I - M + M^2 - M^3) X_D with M = X_D L_off; T = X diag(beta).
//   * The stacked column operand and T enter their MMAs as hi + lo bf16
//     pairs (two accumulating MMAs).
//   * W = T (exp(G) k_hat) and U = T v as M=128 x N=128 x K=64 MMAs; the
//     record is written with 16-byte stores and bulk copies, laid out as the
//     scan's shared-memory image (TcRec).
// One persistent CTA of 16 warps per SM walks the deferred-item list.
#include <algorithm>

#include "kda_chunk_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = kChunk;    // 64
constexpr int D = kHeadDim;  // 128
// ---------------------------------------------------------------------------
// prep
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 512;
constexpr int kLoader = 64;  // issues the TMA loads and the A/L MMA; its warp does no W/U readout
constexpr uint32_t kPrepTmemCols = 256;  // A/L result 0..159; then W 0..127, U 128..255
constexpr int NPAIR = 10;      // (row block br, column block b) pairs with br >= b
constexpr int NST = 16 * NPAIR;  // 160 = N of the stacked A/L MMA
// shared memory plan (offsets from a 1024-aligned base)
constexpr int R_Q = 0;          // bf16 [64][128]
constexpr int R_K = 16384;      // bf16 [64][128]
constexpr int R_V = 32768;      // bf16, two 128B-swizzled [64 rows][64] blocks (MN-major operand)
constexpr int R_G = 49152;      // fp32 [64][128]: g -> G -> l
constexpr int R_BYTES = 81920;
constexpr int P_XL = R_BYTES;             // 32 KB: [q_hat l ; k_hat l] | L fp32 + scratch | E^T, V^T
constexpr int P_BS = P_XL + 32768;        // 40 KB: stacked column operand | inverse scratch, T
constexpr int P_T = P_BS + 16384;         // T operand [64][64] bf16; the MMA reads 16 KB from here
constexpr int P_RQ = P_BS + 40960;        // fp32 [64]: scale / |q_r|
constexpr int P_RK = P_RQ + 256;          // fp32 [64]: 1 / |k_r|
constexpr int P_BETA = P_RK + 256;        // fp32 [64]
constexpr int P_GREF = P_BETA + 256;      // fp32 [5][128]: G at rows 0, 16, 32, 48, 63
constexpr int P_TAU = P_GREF + 5 * 512;   // fp32 [6][128]: exp(G_16br - G_16b), br > b
constexpr int P_QSUM = P_TAU + 6 * 512;   // fp32 [4][128]: per-quarter sums of g
constexpr int P_PSI = P_QSUM + 4 * 512;   // fp32 [4][128]: G_last - G_16b
constexpr int P_FIRST = P_PSI + 4 * 512;  // fp32 [4][128]: g at rows 0, 16, 32, 48
constexpr int P_BAR = P_FIRST + 4 * 512;    // q/k/g barrier, mma barrier, tmem slot, v barrier, metadata
constexpr int P_BS2 = (P_BAR + 64 + 1023) / 1024 * 1024;  // 40 KB: low part of the stacked operand
constexpr int P_E = P_BS2 + 40960;        // 16 KB: E = k_hat exp(G), MN-major [j][d]
constexpr int P_BYTES = P_E + 16384;
constexpr int P_SMEM = P_BYTES + 1024;
static_assert(P_SMEM <= 232448, "prep shared memory");
constexpr int LSTRIDE = 68;               // row stride (floats) of L in shared memory
constexpr float kDiagSpan = 75.0f;        // largest decay inside one 16-token block whose
                                          // diagonal scores the factorised MMA carries
constexpr int MS = 20;                    // row stride (floats) of 16x16 scratch matrices
constexpr int MBLK = 16 * MS;             // floats per 16x16 scratch matrix
static_assert(P_T + 8192 + 16384 <= P_BS + 40960, "T_hi / T_lo operand windows");
static_assert(12 * MBLK * 4 <= P_T - P_BS, "inverse scratch vs T");
static_assert(C * LSTRIDE * 4 + 2 * MBLK * 4 <= 32768, "XL scratch");

__device__ __forceinline__ int tau_index(int br, int b) { return br * (br - 1) / 2 + b; }
// first column of row block br in the stacked A/L result (pairs (br, 0..br) are consecutive)
__device__ __forceinline__ int pair_col0(int br) { return 8 * br * (br + 1); }

struct PrepItem {
    int64_t tok0;
    int valid, h, c;
};

static_assert(32 + sizeof(PrepItem) <= 64, "barrier block");

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

// Raw tiles of one (chunk, head) item through 3-D tensor maps {128, H, T}
// over the [T, H, 128] tensors: q, k (bf16) and g (fp32) as plain row-major
// 128 x 1 x 64 boxes; v (bf16) as two 64 x 1 x 64 boxes with 128-byte
// swizzle, i.e. already the MN-major operand layout of the U MMA.  Rows past
// the end of the tensor arrive as zeros.  q, k and g are loaded as soon as
// the previous item's row pass has consumed them, v after its last MMA.
struct RawMaps {
    CUtensorMap q, k, v, g;
};

// g_bytes: 32 KB for an fp32 g tile, 16 KB for a raw bf16 gate tile
__device__ __forceinline__ void load_qkg(unsigned char *buf, const RawMaps &m, int h, int64_t tok0,
                                         uint64_t *bar, uint32_t g_bytes) {
    mbar_arrive_expect_tx(bar, 16384u + 16384u + g_bytes);
    tma_load_3d(buf + R_Q, &m.q, 0, h, (int)tok0, bar);
    tma_load_3d(buf + R_K, &m.k, 0, h, (int)tok0, bar);
    tma_load_3d(buf + R_G, &m.g, 0, h, (int)tok0, bar);
}

__device__ __forceinline__ void load_v(unsigned char *buf, const RawMaps &m, int h, int64_t tok0,
                                       uint64_t *bar) {
    mbar_arrive_expect_tx(bar, 16384u);
    tma_load_3d(buf + R_V, &m.v, 0, h, (int)tok0, bar);
    tma_load_3d(buf + R_V + 8192, &m.v, 64, h, (int)tok0, bar);
}

// fp32 [rows][128] arrays that are read 8 channels per lane (16 lanes per
// row): channel d is stored at swz(d), i.e. float4 unit u of a row at
// u ^ ((u / 8) % 2), so that each group of 8 lanes covers all 32 banks.
__device__ __forceinline__ int swz(int d) { return d ^ (((d >> 5) & 1) << 2); }

// channels d0 .. d0+7 (d0 a multiple of 8) of a swizzled row
__device__ __forceinline__ void load8s(const float *row, int d0, float (&x)[8]) {
    const int f = ((d0 >> 5) & 1) << 2;
    const float4 a = *reinterpret_cast<const float4 *>(row + (d0 ^ f));
    const float4 b = *reinterpret_cast<const float4 *>(row + ((d0 + 4) ^ f));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Row i of a 16x16 fp32 matrix (row stride lda floats, 16-byte aligned rows).
__device__ __forceinline__ void row16(const float *A, int lda, int i, float (&a)[16]) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        const float4 x = *reinterpret_cast<const float4 *>(A + i * lda + 4 * q4);
        a[4 * q4] = x.x; a[4 * q4 + 1] = x.y; a[4 * q4 + 2] = x.z; a[4 * q4 + 3] = x.w;
    }
}

// Four outputs (row a[], columns 4c4..4c4+3) of a * B, B a 16x16 matrix with
// row stride ldb (floats, 16-byte aligned rows).
__device__ __forceinline__ float4 row4_times(const float (&a)[16], const float *B, int c4,
                                             int ldb = MS) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
        float4 b[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) b[kk] = *reinterpret_cast<const float4 *>(B + (8 * h8 + kk) * ldb + 4 * c4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const float x = a[8 * h8 + kk];
            acc.x = fmaf(x, b[kk].x, acc.x);
            acc.y = fmaf(x, b[kk].y, acc.y);
            acc.z = fmaf(x, b[kk].z, acc.z);
            acc.w = fmaf(x, b[kk].w, acc.w);
        }
    }
    return acc;
}

__device__ __forceinline__ float4 mm16_row4(const float *A, int lda, const float *B, int ldb, int i,
                                            int c4) {
    float a[16];
    row16(A, lda, i, a);
    return row4_times(a, B, c4, ldb);
}

// GATED: maps.g covers the model's raw bf16 gate and beta is unused; the
// gate (GateArgs) is activated on chip.  Otherwise g and beta are activated.
template <bool GATED>
__global__ void __launch_bounds__(kPrepThreads, 1)
    chunk_prep_tc_strong_kernel(const __grid_constant__ RawMaps maps, const float *__restrict__ beta,
                         const GateArgs gate, int n_seqs, int H, float scale, int scan_ctas,
                         int prep_ctas, void *workspace, WsLayout L) {
    constexpr uint32_t kGBytes = GATED ? 16384u : 32768u;
    if (!scan_ctas) {
        griddep_wait();  // the prep (previous kernel) is complete
    } else {
        // the prep's CTAs have all finished (their deferred items listed); the
        // kernel before this one is not waited for, as that would wait for the
        // scan running alongside, which waits for the items listed here
        if (threadIdx.x == 0 && !count_wait(ws_at<const int32_t>(workspace, L.prep_done_off), prep_ctas))
            atomicOr(ws_at<int32_t>(workspace, L.status_off), kStatusTimeout);
        __syncthreads();
    }
    auto beta_of = [&](int64_t tok, int hh) {
        return GATED ? gate_beta(__bfloat162float(
                           reinterpret_cast<const __nv_bfloat16 *>(gate.raw_beta)[tok * H + hh]))
                     : beta[tok * H + hh];
    };
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sXL = sm + P_XL;
    unsigned char *sBS = sm + P_BS;
    unsigned char *sT = sm + P_T;          // T_hi; T_lo follows 8 KB later
    unsigned char *sBS2 = sm + P_BS2;
    float *sB = reinterpret_cast<float *>(sm + P_BETA);
    float *sGref = reinterpret_cast<float *>(sm + P_GREF);
    float *sTau = reinterpret_cast<float *>(sm + P_TAU);
    float *sQsum = reinterpret_cast<float *>(sm + P_QSUM);
    float *sPsi = reinterpret_cast<float *>(sm + P_PSI);
    float *sRq = reinterpret_cast<float *>(sm + P_RQ);
    float *sRk = reinterpret_cast<float *>(sm + P_RK);
    float *sFirst = reinterpret_cast<float *>(sm + P_FIRST);
    unsigned char *sE = sm + P_E;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + P_BAR);
    uint64_t *mbar = full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 1);
    uint64_t *vfull = full + 3;
    PrepItem *sNext = reinterpret_cast<PrepItem *>(sm + P_BAR + 32);  // metadata two items ahead
    int *sBlockFlag = reinterpret_cast<int *>(sm + P_BAR + 56);  // blocks needing exact diagonals
    const __nv_bfloat16 *sQr = reinterpret_cast<const __nv_bfloat16 *>(sm + R_Q);
    const __nv_bfloat16 *sKr = reinterpret_cast<const __nv_bfloat16 *>(sm + R_K);
    float *sG = reinterpret_cast<float *>(sm + R_G);  // g -> G_r - G_16b

    const int32_t *chunk_off = ws_at<const int32_t>(workspace, L.chunk_off_off);
    const int32_t *seq_start = ws_at<const int32_t>(workspace, L.seq_start_off);
    const int32_t *seq_len = ws_at<const int32_t>(workspace, L.seq_len_off);
    int32_t *status = ws_at<int32_t>(workspace, L.status_off);
    const int32_t *list = ws_at<const int32_t>(workspace, L.defer_off);
    const int n_list = *ws_at<const int32_t>(workspace, L.defer_count_off);
    int32_t *ready = ws_at<int32_t>(workspace, L.ready_off);
    // With a scan running alongside (scan_ctas of them), the CTA that finishes
    // last waits for the scan to finish too: whatever follows on the stream
    // waits for this grid, so it then sees the scan's outputs.
    auto finish = [&]() {  // one thread per CTA, at exit
        if (!scan_ctas) return;
        if (atomicAdd(ws_at<int32_t>(workspace, L.strong_done_off), 1) == (int)gridDim.x - 1) {
            griddep_launch_dependents();
            if (!count_wait(ws_at<const int32_t>(workspace, L.scan_done_off), scan_ctas))
                atomicOr(status, kStatusTimeout);
        }
    };
    if ((int)blockIdx.x >= n_list) {
        if (threadIdx.x == 0) finish();
        return;
    }

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) tmem_alloc(tmem_slot, kPrepTmemCols);
    if (tid == 32) {
        mbar_init(full, 1);
        mbar_init(vfull, 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
        *sBlockFlag = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // item metadata runs one item ahead of the loads, which run one item ahead
    // of the compute
    int li = blockIdx.x;  // position in the deferred-item list
    PrepItem cur = prep_item(list[li], H, chunk_off, seq_start, seq_len, n_seqs);
    if (tid == kLoader) {
        load_qkg(sm, maps, cur.h, cur.tok0, full, kGBytes);
        load_v(sm, maps, cur.h, cur.tok0, vfull);
    }
    float beta_cur = tid < cur.valid ? beta_of(cur.tok0 + tid, cur.h) : 0.0f;
    // gate parameters of this thread's key channel (tid % 128) for the current
    // item's head, fetched one item ahead like beta (A_log raw: its exponential
    // is taken where it is used, so the load's latency stalls nothing)
    auto gate_bias = [&](int hh) { return GATED ? gate.dt_bias[hh * D + (tid & (D - 1))] : 0.0f; };
    auto gate_alog = [&](int hh) { return GATED ? gate.a_log[hh] : 0.0f; };
    float bias_cur = gate_bias(cur.h), alog_cur = gate_alog(cur.h);
    PrepItem nxt = cur;
    if (li + (int)gridDim.x < n_list)
        nxt = prep_item(list[li + gridDim.x], H, chunk_off, seq_start, seq_len, n_seqs);

    // phases of the three barriers, and whether a phase is armed but not yet
    // waited for (what must land before the shared memory is released)
    uint32_t fphase = 0, vphase = 0, mphase = 0;
    bool fpend = true, vpend = true, mpend = false;
    bool ok = true;
    for (; li < n_list; li += gridDim.x) {
        const bool has_next = li + (int)gridDim.x < n_list;
        if (!has_next) griddep_launch_dependents();  // last item: the scan may be scheduled
        unsigned char *rec = ws_at<unsigned char>(workspace, L.records_off + ((size_t)cur.c * H + cur.h) * TcRec::bytes);
        const int valid = cur.valid;
        if (tid < C) sB[tid] = tid < valid ? beta_cur : 0.0f;
        float beta_nxt = 0.0f, bias_nxt = 0.0f, alog_nxt = 0.0f;

        if (mbar_wait(full, fphase)) {
            fphase ^= 1;
            fpend = false;
        } else {
            ok = false;
        }
        // rows past the end of the sequence: zero (the tensor map only zero-fills past T)
        for (int i = tid; i < (C - valid) * 16; i += kPrepThreads) {
            const int r = valid + i / 16, c16 = i % 16;
            const uint4 z = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(sm + R_Q + r * 256 + c16 * 16) = z;
            *reinterpret_cast<uint4 *>(sm + R_K + r * 256 + c16 * 16) = z;
            if (!GATED) {  // a raw gate tile is masked row by row on activation instead
                *reinterpret_cast<uint4 *>(sm + R_G + r * 512 + c16 * 32) = z;
                *reinterpret_cast<uint4 *>(sm + R_G + r * 512 + c16 * 32 + 16) = z;
            }
        }
        if (!__syncthreads_and(ok)) {
            ok = false;  // uniform from here on: every thread takes the exit path
            break;
        }

        // 1. cumulative log-decay, one key channel and one 16-row block per
        //    thread: sG receives G_r - G_16b (b = r's block, so <= 0); the
        //    block sums and first-row values then give every reference
        //    quantity of the thread's block: G_16b, G_last - G_16b,
        //    tau(b, b') = exp(G_16b - G_16b'), b' < b, and gC = exp(G_last).
        {
            const int d = tid & (D - 1), qtr = tid >> 7, r0 = 16 * qtr;
            float x[16];
            if (GATED) {  // the model's gate: x = raw + dt_bias, through softplus or sigmoid
                const __nv_bfloat16 *raw = reinterpret_cast<const __nv_bfloat16 *>(sm + R_G);
                const float bias = bias_cur, gs = __expf(alog_cur);
                const bool lb = gate.use_lower_bound != 0;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    x[i] = r0 + i < valid ? gate_decay_fast(__bfloat162float(raw[(r0 + i) * D + d]) + bias,
                                                            gs, gate.lower_bound, lb)
                                          : 0.0f;
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = sG[(r0 + i) * D + d];  // g, plain layout
            }
#pragma unroll
            for (int i = 1; i < 16; ++i) x[i] += x[i - 1];
            {  // a decay span the diagonal block's factors cannot carry
                float span = 0.0f;
#pragma unroll
                for (int i = 1; i < 16; ++i) span = fmaxf(span, fabsf(x[i] - x[0]));
                if (span > kDiagSpan) atomicOr(sBlockFlag, 1 << qtr);
            }
            sQsum[qtr * D + d] = x[15];
            sFirst[qtr * D + d] = x[0];
            const int ds = swz(d);
            __syncthreads();  // every g (or raw gate) value is read: sG is overwritten below
#pragma unroll
            for (int i = 0; i < 16; ++i) sG[(r0 + i) * D + ds] = x[i] - x[0];
            float off = 0.0f, gl = 0.0f, gfirst[3];  // gfirst[b] = G_16b, b < qtr
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float qs = sQsum[b * D + d];
                if (b < qtr) {
                    gfirst[b] = off + sFirst[b * D + d];
                    off += qs;
                }
                gl += qs;
            }
            const float gb = off + x[0];
#pragma unroll
            for (int b = 0; b < 3; ++b)
                if (b < qtr) sTau[tau_index(qtr, b) * D + ds] = __expf(gb - gfirst[b]);
            sGref[qtr * D + ds] = gb;
            sPsi[qtr * D + ds] = gl - gb;
            if (qtr == 3) {
                sGref[4 * D + ds] = gl;
                reinterpret_cast<float *>(rec + TcRec::GC)[d] = __expf(gl);
            }
        }
        if (tid == kLoader) bulk_wait_read();  // the previous item's W/U staging is read
        __syncthreads();
        const int bflags = *sBlockFlag;  // reset once every thread has read it (below)
        // 2. the operands of the A/L MMA, one pass per (row j, 8 channels):
        //    the row norms of q and k (16 lanes per row), l = exp(G_j - G_16bj),
        //    the row operand [q_hat l ; k_hat l], and the stacked column
        //    operand rows of j for every row block br >= bj:
        //    k_hat_j exp(G_16br - G_j) = k_hat_j tau(br, bj) / l_j, with 1 / l_j
        //    clamped at exp(80) on the block diagonal; where l_j < 1e-30 those
        //    entries are taken as exponentials directly.
        //    A thread takes rows r and 63 - r: five column blocks in total.
#pragma unroll  // both rows in one body: their shuffles and exponentials interleave
        for (int it = 0; it < 2; ++it) {
            const int r = it == 0 ? (tid >> 4) : 63 - (tid >> 4), d0 = (tid & 15) * 8, bj = r >> 4;
            float rel8[8], qv[8], kv[8];
            load8s(sG + r * D, d0, rel8);
            unpack8(*reinterpret_cast<const uint4 *>(sQr + r * D + d0), qv);
            unpack8(*reinterpret_cast<const uint4 *>(sKr + r * D + d0), kv);
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                sq = fmaf(qv[t], qv[t], sq);
                sk = fmaf(kv[t], kv[t], sk);
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {  // the 16 lanes of row r
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            const float rq = scale * rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
            if ((tid & 15) == 0) {
                sRq[r] = rq;
                sRk[r] = rk;
            }
            float ql[8], kl[8], l8[8], inv[8], kh[8];
            bool tiny = false;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                l8[t] = __expf(rel8[t]);
                kh[t] = kv[t] * rk;
                ql[t] = qv[t] * rq * l8[t];
                kl[t] = kh[t] * l8[t];
                tiny |= l8[t] < 1e-30f;
                inv[t] = __expf(-rel8[t]);  // 1 / l
            }
            *reinterpret_cast<uint4 *>(sXL + sw128_off(r, d0, 128)) = pack8(ql);
            *reinterpret_cast<uint4 *>(sXL + sw128_off(64 + r, d0, 128)) = pack8(kl);
            // hi + lo bf16 parts: the MMA sees this operand to ~16 bits
            auto emit = [&](int b2, const float (&y)[8]) {
                const uint4 hi = pack8(y);
                float lo[8];
                unpack8(hi, lo);
#pragma unroll
                for (int t = 0; t < 8; ++t) lo[t] = y[t] - lo[t];
                const int row = 16 * (b2 * (b2 + 1) / 2 + bj) + (r & 15);
                *reinterpret_cast<uint4 *>(sBS + sw128_off(row, d0, NST)) = hi;
                *reinterpret_cast<uint4 *>(sBS2 + sw128_off(row, d0, NST)) = pack8(lo);
            };
            if (!__builtin_expect(tiny, 0)) {
                float y[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) y[t] = kh[t] * fminf(inv[t], 5.540622e34f);
                emit(bj, y);
                for (int b2 = bj + 1; b2 < 4; ++b2) {
                    float t8[8];
                    load8s(sTau + tau_index(b2, bj) * D, d0, t8);
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] = kh[t] * t8[t] * inv[t];
                    emit(b2, y);
                }
            } else {  // a decay of more than ~69 inside this 16-row block
                float y[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) y[t] = kh[t] * __expf(fminf(-rel8[t], 80.0f));
                emit(bj, y);
                for (int b2 = bj + 1; b2 < 4; ++b2) {
#pragma unroll
                    for (int t = 0; t < 8; ++t)
                        y[t] = kh[t] * __expf(sGref[b2 * D + swz(d0 + t)] - sGref[bj * D + swz(d0 + t)] - rel8[t]);
                    emit(b2, y);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) *sBlockFlag = 0;
        if (tid == kLoader) {
            tc_fence_after();
            mma_tile<128, NST, 128, 128, NST>(tmem, smem_u32(sXL), smem_u32(sBS), false);
            mma_tile<128, NST, 128, 128, NST>(tmem, smem_u32(sXL), smem_u32(sBS2), true);
            mma_commit(mbar);
        }
        mpend = true;
        // global loads for later items, their latency hidden under the MMA:
        // beta of the next item (used at its start), and the metadata of the
        // item after it, fetched by one thread of a warp that does no TMEM
        // readout (its dependent loads stall only that warp) and handed over
        // in shared memory
        if (has_next && tid < nxt.valid) beta_nxt = beta_of(nxt.tok0 + tid, nxt.h);
        if (GATED && has_next) {
            bias_nxt = gate_bias(nxt.h);
            alog_nxt = gate_alog(nxt.h);
        }
        if (tid == kPrepThreads - 32 && li + 2 * (int)gridDim.x < n_list)
            *sNext = prep_item(list[li + 2 * gridDim.x], H, chunk_off, seq_start, seq_len, n_seqs);

        // While the MMA runs: QG = q_hat exp(G) and KD = k_hat exp(G_last - G)
        // to the record, E = k_hat exp(G) (MN-major [j][d], for W = T E); both
        // exponents are <= 0 and formed from the block-relative G.
#pragma unroll 1
        for (int it = 0; it < 2; ++it) {
            const int r = 32 * it + (tid >> 4), d0 = (tid & 15) * 8, bj = r >> 4;
            float rel8[8], gb8[8], lp8[8], qv[8], kv[8];
            load8s(sG + r * D, d0, rel8);
            load8s(sGref + bj * D, d0, gb8);
            load8s(sPsi + bj * D, d0, lp8);
            unpack8(*reinterpret_cast<const uint4 *>(sQr + r * D + d0), qv);
            unpack8(*reinterpret_cast<const uint4 *>(sKr + r * D + d0), kv);
            const float rq = sRq[r], rk = sRk[r];
            float qg[8], e8[8], kd8[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const float eg = __expf(gb8[t] + rel8[t]), kh = kv[t] * rk;
                qg[t] = qv[t] * rq * eg;
                e8[t] = kh * eg;
                kd8[t] = kh * __expf(lp8[t] - rel8[t]);
            }
            *reinterpret_cast<uint4 *>(rec + TcRec::WQ + sw128_off(64 + r, d0, 128)) = pack8(qg);
            *reinterpret_cast<uint4 *>(sE + sw128_off(r, d0, 64)) = pack8(e8);
            *reinterpret_cast<uint4 *>(rec + TcRec::KD + sw128_off(r, d0, 64)) = pack8(kd8);
        }
        if (mbar_wait(mbar, mphase)) {
            mphase ^= 1;
            mpend = false;
        } else {
            ok = false;
        }
        tc_fence_after();
        if (!__syncthreads_and(ok)) {
            ok = false;  // uniform from here on: every thread takes the exit path
            break;
        }
        // the q, k and g tiles are consumed (unless a block's diagonal scores
        // are recomputed below): the next item's loads go out now
        if (tid == kLoader && has_next && !bflags) load_qkg(sm, maps, nxt.h, nxt.tok0, full, kGBytes);
        fpend = has_next && !bflags;

        // 3. beta-scaled L rows (TMEM lanes 64..127) to shared fp32 by the
        //    warps of lane quarters 2-3; A rows (lanes 0..63) to the record by
        //    warps 4, 5, 8, 9, 12, 13, while the inverse starts as soon as L
        //    is in place.  Row r of block br finds column j of its block pairs
        //    at TMEM column pair_col0(br) + j.
        {
            float *sL = reinterpret_cast<float *>(sXL);
            const int quarter = warp & 3;
            const int r = 32 * (quarter & 1) + lane;  // row inside A (quarters 0,1) or L (2,3)
            const int br = r >> 4;
            const bool lo_pair = (quarter & 1) == 0;  // rows of blocks 0,1: columns [0, 48)
            const int ntile = lo_pair ? 3 : 7;
            const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16);
            if (quarter >= 2) {
                const float bet = sB[r];
                for (int tile = warp >> 2; tile < ntile; tile += 4) {
                    const int c0 = (lo_pair ? 0 : 48) + 16 * tile;
                    float x[16];
                    tmem_ld16(ta + c0, x);
                    tmem_ld_wait();
                    const int j0 = c0 - pair_col0(br);
                    if (j0 < 0 || j0 >= 16 * (br + 1)) continue;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int j = j0 + 4 * c4;
                        float4 y;
                        y.x = (j + 0 < r) ? bet * x[4 * c4 + 0] : 0.0f;
                        y.y = (j + 1 < r) ? bet * x[4 * c4 + 1] : 0.0f;
                        y.z = (j + 2 < r) ? bet * x[4 * c4 + 2] : 0.0f;
                        y.w = (j + 3 < r) ? bet * x[4 * c4 + 3] : 0.0f;
                        *reinterpret_cast<float4 *>(sL + r * LSTRIDE + j) = y;
                    }
                }
                tc_fence_before();
                named_bar_sync(1, 320);
            } else if (warp < 2) {
                named_bar_sync(1, 320);
            } else {
                const int part = (warp >> 2) - 1;  // 0..2
                for (int tile = part; tile < ntile; tile += 3) {
                    const int c0 = (lo_pair ? 0 : 48) + 16 * tile;
                    float x[16];
                    tmem_ld16(ta + c0, x);
                    tmem_ld_wait();
                    const int j0 = c0 - pair_col0(br);
                    if (j0 < 0 || j0 >= 16 * (br + 1)) continue;
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        float y[8];
#pragma unroll
                        for (int t = 0; t < 8; ++t) y[t] = (j0 + 8 * h8 + t <= r) ? x[8 * h8 + t] : 0.0f;
                        *reinterpret_cast<uint4 *>(rec + TcRec::A + sw128_off(r, j0 + 8 * h8, 64)) = pack8(y);
                    }
                }
                // A entries right of a row's block diagonal are zero
                for (int i = 64 * part + 32 * (quarter & 1) + lane; i < C * 8; i += 192) {
                    const int ra = i >> 3, c8 = i & 7;
                    if (c8 >= 2 * ((ra >> 4) + 1))
                        *reinterpret_cast<uint4 *>(rec + TcRec::A + sw128_off(ra, 8 * c8, 64)) = make_uint4(0, 0, 0, 0);
                }
                tc_fence_before();
            }
        }

        // 3b. Blocks whose decay span exceeds kDiagSpan: their diagonal 16 x 16
        //     scores from exact pairwise exponentials (G_r - G_j = the
        //     block-relative sG_r - sG_j), over the MMA's values, in A (record)
        //     and L (shared).  Warp w takes row 16 b + w of each such block, lane
        //     l channels 4l .. 4l+3; lane j - 16 b keeps pair (r, j).  Then the
        //     raw tiles are released to the next item's loads.
        if (bflags) {
            __syncthreads();  // A and L from the MMA are in place
            float *sL = reinterpret_cast<float *>(sXL);
            const int ch = 4 * lane, chs = ch ^ (((ch >> 5) & 1) << 2);  // swizzled float4 unit
            for (int b = 0; b < 4; ++b) {
                if (!((bflags >> b) & 1)) continue;
                const int r = 16 * b + warp;
                const bool live_r = r < valid;
                const float rq = live_r ? sRq[r] : 0.0f, rk = live_r ? sRk[r] : 0.0f;
                float qr[4], kr[4];
                {
                    const uint2 qa = *reinterpret_cast<const uint2 *>(sQr + r * D + ch);
                    const uint2 ka = *reinterpret_cast<const uint2 *>(sKr + r * D + ch);
                    const float2 q0 = unpack2(qa.x), q1 = unpack2(qa.y), k0 = unpack2(ka.x), k1 = unpack2(ka.y);
                    qr[0] = q0.x * rq; qr[1] = q0.y * rq; qr[2] = q1.x * rq; qr[3] = q1.y * rq;
                    kr[0] = k0.x * rk; kr[1] = k0.y * rk; kr[2] = k1.x * rk; kr[3] = k1.y * rk;
                }
                const float4 gr = *reinterpret_cast<const float4 *>(sG + r * D + chs);
                const float bet = sB[r];
                float av = 0.0f, lv = 0.0f;
                for (int j = 16 * b; j <= r; ++j) {
                    const bool live_j = j < valid;
                    const float rkj = live_j ? sRk[j] : 0.0f;
                    const uint2 kb = *reinterpret_cast<const uint2 *>(sKr + j * D + ch);
                    const float2 k0 = unpack2(kb.x), k1 = unpack2(kb.y);
                    const float4 gj = *reinterpret_cast<const float4 *>(sG + j * D + chs);
                    const float e0 = __expf(gr.x - gj.x), e1 = __expf(gr.y - gj.y);
                    const float e2 = __expf(gr.z - gj.z), e3 = __expf(gr.w - gj.w);
                    const float w0 = k0.x * rkj * e0, w1 = k0.y * rkj * e1, w2 = k1.x * rkj * e2,
                                w3 = k1.y * rkj * e3;
                    float a = qr[0] * w0, l = kr[0] * w0;
                    a = fmaf(qr[1], w1, a); l = fmaf(kr[1], w1, l);
                    a = fmaf(qr[2], w2, a); l = fmaf(kr[2], w2, l);
                    a = fmaf(qr[3], w3, a); l = fmaf(kr[3], w3, l);
                    a = warp_sum(a);
                    l = warp_sum(l);
                    if (lane == j - 16 * b) {
                        av = a;
                        lv = j < r ? bet * l : 0.0f;
                    }
                }
                if (lane < 16) {  // columns 16 b .. 16 b + 15 of row r
                    const int j = 16 * b + lane;
                    sL[r * LSTRIDE + j] = lv;
                    *reinterpret_cast<__nv_bfloat16 *>(rec + TcRec::A + sw128_off(r, j, 64)) =
                        __float2bfloat16_rn(j <= r ? av : 0.0f);
                }
            }
            if (tid == 0) atomicOr(status, kExactDecay);
            __syncthreads();  // the raw tiles are read: the next item's loads go out
            if (tid == kLoader && has_next) load_qkg(sm, maps, nxt.h, nxt.tok0, full, kGBytes);
            fpend = has_next;
        }

        // 4. X = (I + L)^-1 with L strictly lower (beta-scaled rows), in 16x16
        //    blocks, and T = X diag(beta) written straight into the bf16 hi + lo
        //    operand (K-major [i][j]) at sT.  Blocked forward substitution:
        //      A: per diagonal block a, forward substitution with (I + L_aa),
        //         one right-hand side per lane: the unit vectors give
        //         X_aa = (I + L_aa)^-1, the columns of L_ab (b < a) give
        //         M_ab = X_aa L_ab (160 lanes, no barriers);
        //      B: X_10 = -M_10 X_00, X_21 = -M_21 X_11, X_32 = -M_32 X_22,
        //         C30 = M_32 M_20 - M_30, C31 = M_32 M_21 - M_31; the
        //         diagonal blocks of T;
        //      C: X_20 = -(M_20 X_00 + M_21 X_10), X_31 = -(M_31 X_11 + M_32 X_21),
        //         X_30 = C30 X_00 + C31 X_10 (= -(M_30 X_00 + M_31 X_10 + M_32 X_20));
        //         zeros above the block diagonal.
        //    Stages B and C give each thread one (row, 4 columns) slot.
        {
            const float *sL = reinterpret_cast<const float *>(sXL);
            float *XD = reinterpret_cast<float *>(sBS);    // X_aa, a = 0..3
            float *Mb = XD + 4 * MBLK;                     // M_ab, pairs p = 0..5
            float *Cb = Mb + 6 * MBLK;                     // C30, C31
            float *Xo = reinterpret_cast<float *>(sXL) + C * LSTRIDE;  // X_10, X_21
            // Block pairs (a, b), a > b, index p: (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
            auto pair_a = [](int p_) { return p_ < 1 ? 1 : (p_ < 3 ? 2 : 3); };
            // T block (a, b), rows i, columns 4c4..4c4+3 from X values x
            auto put_t = [&](int a, int b, int i, int c4, float4 x) {
                const int row = 16 * a + i, col = 16 * b + 4 * c4;
                const float4 bt = *reinterpret_cast<const float4 *>(sB + col);
                const float y0 = x.x * bt.x, y1 = x.y * bt.y, y2 = x.z * bt.z, y3 = x.w * bt.w;
                const uint32_t h01 = pack2(y0, y1), h23 = pack2(y2, y3);
                const float2 f01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&h01));
                const float2 f23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&h23));
                const uint32_t off = sw128_off(row, col, 64);
                *reinterpret_cast<uint2 *>(sT + off) = make_uint2(h01, h23);
                *reinterpret_cast<uint2 *>(sT + 8192 + off) =
                    make_uint2(pack2(y0 - f01.x, y1 - f01.y), pack2(y2 - f23.x, y3 - f23.y));
            };
            const int sidx = warp < 4 ? warp : (warp == 6 ? 4 : 5);  // stage A: warps 0, 1, 2, 3, 6
            if (sidx < 5) {
                const int sl = 32 * sidx + lane;
                const bool unit = sl < 64;
                const int p_ = unit ? 0 : (sl - 64) >> 4;
                const int a = unit ? sl >> 4 : pair_a(p_);
                const int b = unit ? a : p_ - a * (a - 1) / 2;
                const int c = sl & 15, o = 16 * a;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float lr[16];
                    row16(sL + o, LSTRIDE, o + r, lr);
                    const float rhs = unit ? (r == c ? 1.0f : 0.0f) : sL[(o + r) * LSTRIDE + 16 * b + c];
                    // two partial sums shorten the dependent chain
                    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
                    for (int m2 = 0; m2 < r; ++m2) {
                        if (m2 & 1) a1 = fmaf(lr[m2], x[m2], a1);
                        else a0 = fmaf(lr[m2], x[m2], a0);
                    }
                    x[r] = rhs - (a0 + a1);
                }
                float *dst = unit ? XD + a * MBLK : Mb + p_ * MBLK;
#pragma unroll
                for (int r = 0; r < 16; ++r) dst[r * MS + c] = x[r];
            }
            __syncthreads();
            {
                const int q_ = tid >> 6, ii = (tid >> 2) & 15, c4 = tid & 3;
                if (q_ < 3) {  // X_{q+1,q} = -M_{q+1,q} X_qq
                    const int pm = q_ == 0 ? 0 : (q_ == 1 ? 2 : 5);
                    float4 x = mm16_row4(Mb + pm * MBLK, MS, XD + q_ * MBLK, MS, ii, c4);
                    x = make_float4(-x.x, -x.y, -x.z, -x.w);
                    if (q_ < 2) *reinterpret_cast<float4 *>(Xo + q_ * MBLK + ii * MS + 4 * c4) = x;
                    put_t(q_ + 1, q_, ii, c4, x);
                } else if (q_ < 5) {  // C30 = M_32 M_20 - M_30, C31 = M_32 M_21 - M_31
                    const int k_ = q_ - 3;
                    float4 x = mm16_row4(Mb + 5 * MBLK, MS, Mb + (k_ == 0 ? 1 : 2) * MBLK, MS, ii, c4);
                    const float4 m = *reinterpret_cast<const float4 *>(Mb + (3 + k_) * MBLK + ii * MS + 4 * c4);
                    *reinterpret_cast<float4 *>(Cb + k_ * MBLK + ii * MS + 4 * c4) =
                        make_float4(x.x - m.x, x.y - m.y, x.z - m.z, x.w - m.w);
                } else {  // diagonal blocks of T: 256 slots over the last 192 threads
                    for (int sl = tid - 320; sl < 256; sl += 192) {
                        const int a = sl >> 6, i = (sl >> 2) & 15, cc = sl & 3;
                        put_t(a, a, i, cc, *reinterpret_cast<const float4 *>(XD + a * MBLK + i * MS + 4 * cc));
                    }
                }
            }
            __syncthreads();
            {
                const int q_ = tid >> 6, ii = (tid >> 2) & 15, c4 = tid & 3;
                if (q_ < 3) {
                    float a16[16];
                    float4 x, y;
                    if (q_ == 0) {         // X_20 = -(M_20 X_00 + M_21 X_10)
                        row16(Mb + 1 * MBLK, MS, ii, a16);
                        x = row4_times(a16, XD, c4);
                        row16(Mb + 2 * MBLK, MS, ii, a16);
                        y = row4_times(a16, Xo, c4);
                        x = make_float4(-(x.x + y.x), -(x.y + y.y), -(x.z + y.z), -(x.w + y.w));
                        put_t(2, 0, ii, c4, x);
                    } else if (q_ == 1) {  // X_31 = -(M_31 X_11 + M_32 X_21)
                        row16(Mb + 4 * MBLK, MS, ii, a16);
                        x = row4_times(a16, XD + MBLK, c4);
                        row16(Mb + 5 * MBLK, MS, ii, a16);
                        y = row4_times(a16, Xo + MBLK, c4);
                        x = make_float4(-(x.x + y.x), -(x.y + y.y), -(x.z + y.z), -(x.w + y.w));
                        put_t(3, 1, ii, c4, x);
                    } else {               // X_30 = C30 X_00 + C31 X_10
                        row16(Cb, MS, ii, a16);
                        x = row4_times(a16, XD, c4);
                        row16(Cb + MBLK, MS, ii, a16);
                        y = row4_times(a16, Xo, c4);
                        put_t(3, 0, ii, c4, make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w));
                    }
                } else {  // zeros above the block diagonal: 6 blocks x 16 rows x 2 chunks x hi, lo
                    for (int sl = tid - 192; sl < 384; sl += 320) {
                        const int pz = sl >> 6, i = (sl >> 2) & 15, h = (sl >> 1) & 1, hl = sl & 1;
                        const int a = pz < 3 ? 0 : (pz < 5 ? 1 : 2);
                        const int b = pz < 3 ? pz + 1 : (pz < 5 ? pz - 1 : 3);
                        *reinterpret_cast<uint4 *>(sT + hl * 8192 + sw128_off(16 * a + i, 16 * b + 8 * h, 64)) =
                            make_uint4(0, 0, 0, 0);
                    }
                }
            }
        }
        __syncthreads();

        // 5. W = T E, U = T V (B operands MN-major: E from the row pass, V as
        //    loaded); hi + lo parts of T.  The v tile was requested at the end
        //    of the previous item; rows past the sequence end are zeroed.
        if (mbar_wait(vfull, vphase)) {
            vphase ^= 1;
            vpend = false;
        } else {
            ok = false;
        }
        for (int i = tid; i < (C - valid) * 16; i += kPrepThreads) {
            const int r = valid + i / 16, c16 = i % 16;
            *reinterpret_cast<uint4 *>(sm + R_V + (c16 >> 3) * 8192 + r * 128 + (c16 & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) {
            ok = false;  // uniform from here on: every thread takes the exit path
            break;
        }
        if (tid == 0) {
            tc_fence_after();
            mma_tile<128, 128, 64, 128, 64, false, true>(tmem + 0, smem_u32(sT), smem_u32(sE), false);
            mma_tile<128, 128, 64, 128, 64, false, true>(tmem + 0, smem_u32(sT + 8192), smem_u32(sE), true);
            mma_tile<128, 128, 64, 128, 64, false, true>(tmem + 128, smem_u32(sT), smem_u32(sm + R_V), false);
            mma_tile<128, 128, 64, 128, 64, false, true>(tmem + 128, smem_u32(sT + 8192), smem_u32(sm + R_V), true);
            mma_commit(mbar);
        }
        mpend = true;
        if (mbar_wait(mbar, mphase)) {
            mphase ^= 1;
            mpend = false;
        } else {
            ok = false;
        }
        tc_fence_after();
        // v is consumed: the next item's v load goes out
        if (tid == kLoader && has_next) load_v(sm, maps, nxt.h, nxt.tok0, vfull);
        vpend = has_next;

        // 6. W rows (WQ rows 0..63) and U: TMEM lanes 0..63 -> shared memory
        //    (sXL, free since the T conversion) in the record's own layout ->
        //    three bulk copies to the record.  U rows are stored with their
        //    16-byte chunks rotated (chunk c of row i at c ^ ((i / 2) % 4)),
        //    which keeps these writes and the scan's reads free of bank
        //    conflicts.  The staging area is reused once the copies have read
        //    it (checked before the next row pass).
        if ((warp & 3) < 2) {
            const int i = 32 * (warp & 3) + lane, part = warp >> 2;
            const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
            float x[32];
            tmem_ld32(ta + 32 * part, x);
            tmem_ld_wait();
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float y[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t];
                *reinterpret_cast<uint4 *>(sXL + sw128_off(i, 32 * part + 8 * c8, 64)) = pack8(y);
            }
            tmem_ld32(ta + 128 + 32 * part, x);
            tmem_ld_wait();
            unsigned char *ub = sXL + 16384 + part * TcRec::UBLK + i * 64;
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float y[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t];
                *reinterpret_cast<uint4 *>(ub + ((c8 ^ ((i >> 1) & 3)) << 4)) = pack8(y);
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) {
            ok = false;  // uniform from here on: every thread takes the exit path
            break;
        }
        if (tid == kLoader) {
            bulk_s2g(rec + TcRec::WQ, sXL, 8192);                  // W, key columns 0..63
            bulk_s2g(rec + TcRec::WQ + 16384, sXL + 8192, 8192);   // W, key columns 64..127
            bulk_s2g(rec + TcRec::U, sXL + 16384, 4 * TcRec::UBLK);
            bulk_commit();
            bulk_wait_all();  // the record is complete (the other parts precede the barrier above)
            flag_publish(ready + (size_t)cur.c * H + cur.h);
        }
        cur = nxt;
        if (li + 2 * (int)gridDim.x < n_list) nxt = *sNext;
        beta_cur = beta_nxt;
        bias_cur = bias_nxt;
        alog_cur = alog_nxt;
    }
    if (tid == kLoader) bulk_wait_all();  // the last record's W and U are written
    if (!ok) {
        if (tid == kLoader) {
            atomicOr(status, kStatusTimeout);
            // let copies and MMAs still in flight land before the shared memory
            // and the TMEM are released
            if (fpend) mbar_wait(full, fphase, 400000000LL);
            if (vpend) mbar_wait(vfull, vphase, 400000000LL);
            if (mpend) mbar_wait(mbar, mphase, 400000000LL);
        }
        __syncthreads();
    }
    if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
    if (tid == kLoader) finish();
}

}  // namespace

void preload_chunk_tc_strong_kernels() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, chunk_prep_tc_strong_kernel<true>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, chunk_prep_tc_strong_kernel<false>) != cudaSuccess)
        cudaGetLastError();
}

cudaError_t launch_chunk_prep_tc_strong(const void *q, const void *k, const void *v,
                                        const float *g, const float *beta, const GateArgs *gate,
                                        int n_seqs, int64_t total_tokens, int H, float scale,
                                        int scan_ctas, int prep_ctas, void *workspace,
                                        cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, TcRec::bytes);
    const int64_t items_max = max_chunks(total_tokens, n_seqs) * (int64_t)H;
    const int grid = (int)std::min<int64_t>(items_max, (int64_t)sm_count());
    if (grid <= 0) return cudaSuccess;
    RawMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (total_tokens > 0) {
        if (!encode_rows(&maps.q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens) ||
            !encode_rows(&maps.k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens) ||
            !encode_rows(&maps.v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens, true) ||
            !(gate ? encode_rows(&maps.g, gate->raw_gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H,
                                 total_tokens)
                   : encode_rows(&maps.g, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, total_tokens)))
            return cudaErrorInvalidValue;
    }
    GateArgs ga;
    memset(&ga, 0, sizeof(ga));
    if (gate) ga = *gate;
    auto kern = gate ? chunk_prep_tc_strong_kernel<true> : chunk_prep_tc_strong_kernel<false>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    const cudaError_t e = launch_dependent(kern, dim3(grid), dim3(kPrepThreads), P_SMEM, stream,
                                           maps, beta, ga, n_seqs, H, scale, scan_ctas, prep_ctas,
                                           workspace, L);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kda
