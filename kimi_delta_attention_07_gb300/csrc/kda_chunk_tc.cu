// Tensor-core (tcgen05) chunked KDA for bf16 inputs: bf16 MMA operands, fp32
// accumulation in TMEM, fp32 recurrent state.
//
// Same two phases as the fp32 path (chunked form of the Ascend model file's
// _torch_chunk_kda), with every dense contraction on the 5th-generation
// tensor cores.
//
// prep -- persistent, two CTAs (8 warps each) per SM walking the (chunk,
// head) items, so that one CTA's barrier-separated phases overlap the
// other's; the raw q, k, v tiles of an item arrive by TMA, g as a register
// slice per thread fetched during the previous item:
//   * q_hat = scale * l2norm(q), k_hat = l2norm(k) (fp32), G = cumsum(g).
//   * Every exponential is referenced to the chunk's middle token:
//     x_r = exp(G_r - G_31) per key channel, so that
//     exp(G_r - G_j) = x_r / x_j, exp(G_r) = x_r exp(G_31) and
//     exp(G_63 - G_j) = exp(G_63 - G_31) / x_j.  A chunk with some
//     |G_r - G_31| > 80 does not fit these factors; it is listed in the
//     workspace and computed by the strong-decay prep (kda_chunk_tc_strong.cu,
//     per-16-token references) right after.
//   * Causal scores A[r,j] and the interaction matrix L[r,j] come from ONE
//     M=128 x N=64 x K=128 MMA: A operand [q_hat x ; k_hat x] (formed in
//     place over the raw q, k tiles, which TMA delivers in that operand's
//     layout), B operand k_hat / x as a hi + lo bf16 pair.
//   * X = (I + beta L)^-1 blockwise in fp32: 16x16 diagonal blocks by
//     forward substitution (one column per lane), the rest as
//     (I - M + M^2 - M^3) X_D with M = X_D L_off; T = X diag(beta), entered
//     into its MMAs as a hi + lo bf16 pair, which keeps the WY transform
//     accurate when keys are strongly correlated and the later subtraction
//     U - W S cancels.
//   * W = T (exp(G) k_hat) and U = T v as M=128 x N=128 x K=64 MMAs whose A
//     operand is [T ; scratch] (rows 64..127 unused), so each thread of
//     TMEM lanes 0..63 holds whole rows of W and U.
//   * Record laid out as the scan's shared-memory image (128-byte-swizzled
//     K-major operands), see TcRec; W and U leave by bulk copies.
//
// scan, one CTA per (sequence, head, 32 value columns), 4 warps, records in a
// 3-stage cp.async.bulk ring:
//     D1  = WQ * S            (M=128, N=32, K=128)  rows 0..63: W S
//     Vn  = U - D1[0:64]      (fp32, written as a bf16 MN-major operand)
//     D1 += [* ; A] * Vn      (rows 64..127 become o = QG S + A Vn)
//     D3  = KD^T * Vn         (M=128, N=32, K=64; KD as an MN-major operand)
//     S   = diag(gC) S + D3   (fp32, one key row per thread, in registers)
//   The 128-row A operand of the second MMA starts 8 KB before the A tile in
//   the staged record (its rows 0..63 are the tail of KD and only feed D1
//   rows that were already consumed).  D1 is double-buffered in TMEM so that
//   the output rows of a chunk are stored while the next chunk's first MMA
//   runs; only the MMA-issuing thread waits for a stage before that MMA.
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
constexpr int kPrepThreads = 256;
constexpr int kPrepMinBlocks = 2;        // two CTAs per SM overlap each other's phases
// the thread that copies W and U to the record and raises its ready flag,
// with a scan running alongside: a lane of warp 4, whose warps finish the
// transform pass ahead of warps 0-3 (without one, thread 0 copies them)
constexpr int kStoreThread = 128;
constexpr uint32_t kPrepTmemCols = 256;  // A/L result 0..63; then W 0..127, U 128..255
constexpr float kLog2e = 1.4426950408889634f;
// Largest |G_r - G_ref| (natural log units, ref = the reference row of r's
// half) the factorised exponentials take: both factors stay inside fp32 /
// bf16 range.  Chunks beyond it are deferred to the strong-decay prep.
constexpr float kRelLimit2 = 80.0f * kLog2e;
constexpr int NCOL = 96;  // column-operand rows of the A/L MMA: 32 per (column half, reference)
// shared memory plan (offsets from a 1024-aligned base)
constexpr int P_XL = 0;             // 32 KB: raw [q ; k] (TMA) -> [q_hat x ; k_hat x]
constexpr int P_COL = 32768;        // 48 KB: B operand of the A/L MMA, 2 NCOL rows: the
                                    // column operand's hi part (rows 0..95), then its lo part
constexpr int P_E = 81920;          // 16 KB: E = k_hat exp(G), MN-major [j][d]
constexpr int P_RQ = 98304;         // fp32 [64]: scale / |q_r|
constexpr int P_RK = P_RQ + 256;    // fp32 [64]: 1 / |k_r|
constexpr int P_BETA = P_RK + 256;  // fp32 [64]
constexpr int P_QS = P_BETA + 256;  // fp32 [8][128]: per-octet sums of g (log2 units)
constexpr int P_BAR = P_QS + 4096;  // q/k barrier, v barrier, mma barrier, tmem slot, metadata
constexpr int P_BYTES = P_BAR + 128;
constexpr int P_SMEM = P_BYTES + 1024;
// reuse of [0, 64 KB) once the A/L MMA has read its operands
constexpr int P_L = 0;              // fp32 [64][LSTRIDE]: beta-scaled L
constexpr int P_SCR = 17408;        // inverse scratch: X_aa and M_ab (10 16x16 fp32 blocks);
                                    // C30, C31, X_10, X_21 reuse L's space once L is consumed
constexpr int P_T = 32768;          // T operand: [T_hi ; T_hi] then [T_lo ; T_lo], 16 KB each
constexpr int P_V = 65536;          // 16 KB: v, MN-major (two 64-column boxes), loaded after A/L
constexpr int P_STAGE = 32768;      // W and U staged for the record after the W/U MMA
constexpr int LSTRIDE = 68;         // row stride (floats) of L in shared memory
constexpr int MS = 20;              // row stride (floats) of 16x16 scratch matrices
constexpr int MBLK = 16 * MS;       // floats per 16x16 scratch matrix
static_assert(P_SMEM * kPrepMinBlocks + 2048 <= 233472, "two prep CTAs per SM");
static_assert(P_L + C * LSTRIDE * 4 <= P_SCR && P_SCR + 10 * MBLK * 4 <= P_XL + 32768 &&
                  4 * MBLK * 4 <= C * LSTRIDE * 4,
              "L and inverse scratch inside the q/k region");
static_assert(P_T + 32768 <= P_V && P_V + 16384 == P_E && P_STAGE + 32768 <= P_E,
              "T and staging below [v | E], one N = 256 operand of four 8 KB column blocks");
static_assert(P_COL + 2 * NCOL * 256 <= P_E, "column operand");

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
// over the [T, H, 128] bf16 tensors, as 64-channel x 1 x 64-token boxes with
// 128-byte swizzle: q and k land as the row blocks of the A/L MMA's K-major
// A operand ([q ; k], 128 rows), v as the MN-major B operand of U = T V.
// Rows past the end of the tensor arrive as zeros.
struct RawMaps {
    CUtensorMap q, k, v;
    CUtensorMap g;  // g fp32, or the raw bf16 gate: only prefetched into L2
};

__device__ __forceinline__ void load_qk(unsigned char *sm, const RawMaps &m, int h, int64_t tok0,
                                        uint64_t *bar) {
    mbar_arrive_expect_tx(bar, 32768u);
    tma_load_3d(sm + P_XL, &m.q, 0, h, (int)tok0, bar);           // q, channels 0..63
    tma_load_3d(sm + P_XL + 8192, &m.k, 0, h, (int)tok0, bar);    // k, channels 0..63
    tma_load_3d(sm + P_XL + 16384, &m.q, 64, h, (int)tok0, bar);  // q, channels 64..127
    tma_load_3d(sm + P_XL + 24576, &m.k, 64, h, (int)tok0, bar);  // k, channels 64..127
}

__device__ __forceinline__ void load_v(unsigned char *sm, const RawMaps &m, int h, int64_t tok0,
                                       uint64_t *bar) {
    mbar_arrive_expect_tx(bar, 16384u);
    tma_load_3d(sm + P_V, &m.v, 0, h, (int)tok0, bar);
    tma_load_3d(sm + P_V + 8192, &m.v, 64, h, (int)tok0, bar);
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

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16 bytes of a global tensor through the non-coherent path, issued where
// it stands (the inputs are read-only for the kernel's lifetime); the value
// is consumed much later, so the load's latency hides under other phases.
__device__ __forceinline__ uint4 ldg16_now(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg8_now(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// g of one thread's (8 rows, 4 channels) slice, fetched into registers: the
// activated fp32 g, or the model's raw bf16 gate (activated with the
// cumulative sum).  Rows past the sequence end read nothing (zero decay).
template <bool GATED>
struct GSlice {
    uint4 v[8];
};
template <>
struct GSlice<true> {
    uint2 v[8];
};

template <bool GATED>
__device__ __forceinline__ void load_gslice(GSlice<GATED> &s, const float *g, const GateArgs &gate,
                                            int64_t tok0, int valid, int r0, int h, int H, int d) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = r0 + i;
        const int64_t off = ((tok0 + r) * H + h) * (int64_t)D + d;
        if constexpr (GATED)
            s.v[i] = r < valid ? ldg8_now(reinterpret_cast<const __nv_bfloat16 *>(gate.raw_gate) + off)
                               : make_uint2(0u, 0u);
        else
            s.v[i] = r < valid ? ldg16_now(g + off) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Main prep: every (chunk, head) item whose decay fits one chunk-wide
// exponential reference; the others are listed for the strong-decay prep.
// GATED: the raw gate of the model is activated on chip (gate.raw_gate /
// raw_beta are read like g / beta).  Otherwise g and beta are the activated
// fp32 inputs.
template <bool GATED>
__global__ void __launch_bounds__(kPrepThreads, kPrepMinBlocks)
    chunk_prep_tc_kernel(const __grid_constant__ RawMaps maps, const float *__restrict__ g,
                         const float *__restrict__ beta, const GateArgs gate, int n_seqs, int H,
                         float scale, int scan_ctas, void *workspace, WsLayout L) {
    // the chunk index (previous kernel) is complete; launched after a scan
    // that runs alongside, whose completion is not waited for, the index
    // finished before that scan was let go
    if (!scan_ctas) griddep_wait();
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sXL = sm + P_XL;
    unsigned char *sE = sm + P_E;
    unsigned char *sT = sm + P_T;  // [T_hi ; T_hi], then [T_lo ; T_lo] 16 KB later
    float *sRq = reinterpret_cast<float *>(sm + P_RQ);
    float *sRk = reinterpret_cast<float *>(sm + P_RK);
    float *sB = reinterpret_cast<float *>(sm + P_BETA);
    float *sQS = reinterpret_cast<float *>(sm + P_QS);
    uint64_t *full_qk = reinterpret_cast<uint64_t *>(sm + P_BAR);
    uint64_t *full_v = full_qk + 1;
    uint64_t *mbar = full_qk + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(full_qk + 3);
    PrepItem *sNext = reinterpret_cast<PrepItem *>(sm + P_BAR + 32);  // metadata two items ahead
    int *sFirst = reinterpret_cast<int *>(sm + P_BAR + 64);            // this CTA's first item
    int *sPub = sFirst + 1;  // store thread: the item whose record waits for its ready flag, or -1
    const int store_tid = scan_ctas ? kStoreThread : 0;

    const int32_t *chunk_off = ws_at<const int32_t>(workspace, L.chunk_off_off);
    const int32_t *seq_start = ws_at<const int32_t>(workspace, L.seq_start_off);
    const int32_t *seq_len = ws_at<const int32_t>(workspace, L.seq_len_off);
    int32_t *status = ws_at<int32_t>(workspace, L.status_off);
    int32_t *defer_count = ws_at<int32_t>(workspace, L.defer_count_off);
    int32_t *defer_list = ws_at<int32_t>(workspace, L.defer_off);
    {  // clear the scan's row-sum exchange ring (its tags) for this call
        uint4 *ring = ws_at<uint4>(workspace, L.epi_part_off);
        const int n16 = min(n_seqs * H, kEpiPairs) * kEpiRing * 4 * C / 2;
        for (int i = blockIdx.x * kPrepThreads + threadIdx.x; i < n16; i += gridDim.x * kPrepThreads)
            ring[i] = make_uint4(0, 0, 0, 0);
    }
    const int n_items = chunk_off[n_seqs] * H;
    // Items go out in (chunk, head) order as CTAs ask for them (two at the
    // start, then one per item, two items ahead), so that records are written
    // chunk by chunk whichever CTAs are resident; each record's ready flag is
    // raised once it is written (the previous item's, when the next item finds
    // its bulk copies done; the last one's at exit).
    if (threadIdx.x == 0) {
        *sFirst = atomicAdd(ws_at<int32_t>(workspace, L.item_ctr_off), 2);
        *sPub = -1;
    }
    __syncthreads();
    const int first = *sFirst;
    // this CTA's writes (records, deferred-item list) are done: with a scan
    // running alongside, the strong-decay prep counts finished CTAs instead of
    // waiting for this grid
    int32_t *prep_done = ws_at<int32_t>(workspace, L.prep_done_off);
    if (first >= n_items) {
        if (threadIdx.x == 0) count_release(prep_done);
        return;
    }
    // "no item" is an item of no rows (valid = 0, token 0, head 0): its loads
    // (a tile that is read but never used, no g or beta) go out like a real
    // item's, so that nothing below branches on whether there is a next item
    auto no_item = []() {
        PrepItem p;
        p.tok0 = 0;
        p.valid = 0;
        p.h = 0;
        p.c = 0;
        return p;
    };
    auto take_item = [&]() {  // one thread
        const int id = atomicAdd(ws_at<int32_t>(workspace, L.item_ctr_off), 1);
        return id < n_items ? prep_item(id, H, chunk_off, seq_start, seq_len, n_seqs) : no_item();
    };
    auto publish = [&]() {  // the store thread, once the copies of the pending record are done
        const int pub = *sPub;
        if (pub >= 0) flag_publish(ws_at<int32_t>(workspace, L.ready_off) + pub);
        *sPub = -1;
    };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // transform-pass slice of this thread: key channels d .. d+3 of the 8
    // rows r0 .. r0+7 (one warp = all 128 channels of 8 rows)
    const int d = 4 * lane, r0 = 8 * warp;
    // its byte offsets in 128-byte-swizzled K-major tiles: K-block, chunk, half
    const int kb = lane >> 4, cw = (lane & 15) >> 1, hb = (lane & 1) * 8;
    if (warp == 0) tmem_alloc(tmem_slot, kPrepTmemCols);
    if (tid == 32) {
        mbar_init(full_qk, 1);
        mbar_init(full_v, 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto beta_of = [&](int64_t tok, int hh) {
        return GATED ? gate_beta(__bfloat162float(
                           reinterpret_cast<const __nv_bfloat16 *>(gate.raw_beta)[tok * H + hh]))
                     : beta[tok * H + hh];
    };
    PrepItem cur = prep_item(first, H, chunk_off, seq_start, seq_len, n_seqs);
    if (tid == 0) load_qk(sm, maps, cur.h, cur.tok0, full_qk);
    GSlice<GATED> gs;
    load_gslice<GATED>(gs, g, gate, cur.tok0, cur.valid, r0, cur.h, H, d);
    float beta_cur = tid < cur.valid ? beta_of(cur.tok0 + tid, cur.h) : 0.0f;
    float4 bias_cur = make_float4(0.f, 0.f, 0.f, 0.f);
    float alog_cur = 0.0f;
    if (GATED) {
        bias_cur = *reinterpret_cast<const float4 *>(gate.dt_bias + cur.h * D + d);
        alog_cur = gate.a_log[cur.h];
    }
    PrepItem nxt = first + 1 < n_items ? prep_item(first + 1, H, chunk_off, seq_start, seq_len, n_seqs)
                                       : no_item();

    uint32_t qkphase = 0, vphase = 0, mphase = 0;
    bool qkpend = true, vpend = false, mpend = false;
    bool ok = true;
    for (;;) {
        if (!nxt.valid) griddep_launch_dependents();  // last item: the next kernel may be scheduled
        // the next item's tiles and beta into L2 now, so that its loads (issued
        // late in this item, where their shared memory and registers free up)
        // find them there
        // (from warp 2: a release of a record's flag by the thread that copies
        // the records would wait for these)
        if (tid == 64 && nxt.valid) {
            tma_prefetch_3d(&maps.q, 0, nxt.h, (int)nxt.tok0);
            tma_prefetch_3d(&maps.q, 64, nxt.h, (int)nxt.tok0);
            tma_prefetch_3d(&maps.k, 0, nxt.h, (int)nxt.tok0);
            tma_prefetch_3d(&maps.k, 64, nxt.h, (int)nxt.tok0);
            tma_prefetch_3d(&maps.v, 0, nxt.h, (int)nxt.tok0);
            tma_prefetch_3d(&maps.v, 64, nxt.h, (int)nxt.tok0);
            tma_prefetch_3d(&maps.g, 0, nxt.h, (int)nxt.tok0);
        } else if (tid >= 192 && tid - 192 < nxt.valid) {
            const int64_t bt = (nxt.tok0 + (tid - 192)) * H + nxt.h;
            prefetch_l2(GATED ? (const void *)(reinterpret_cast<const __nv_bfloat16 *>(gate.raw_beta) + bt)
                              : (const void *)(beta + bt));
        }
        unsigned char *rec = ws_at<unsigned char>(workspace, L.records_off + ((size_t)cur.c * H + cur.h) * TcRec::bytes);
        const int valid = cur.valid;
        if (tid < C) sB[tid] = tid < valid ? beta_cur : 0.0f;

        // 1. cumulative log2-decay over this thread's 8 rows, per channel, in
        //    registers: pre_i = log2(e) * sum of g over rows r0 .. r0+i.  The
        //    8-row total goes to shared memory.
        float4 pre[8];
        {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const float gsc = GATED ? __expf(alog_cur) : 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float4 gv;
                if constexpr (GATED) {
                    const float2 a = unpack2(gs.v[i].x), b = unpack2(gs.v[i].y);
                    const bool live = r0 + i < valid;
                    const float lb = gate.lower_bound;
                    const bool ulb = gate.use_lower_bound != 0;
                    gv.x = live ? gate_decay_fast(a.x + bias_cur.x, gsc, lb, ulb) : 0.0f;
                    gv.y = live ? gate_decay_fast(a.y + bias_cur.y, gsc, lb, ulb) : 0.0f;
                    gv.z = live ? gate_decay_fast(b.x + bias_cur.z, gsc, lb, ulb) : 0.0f;
                    gv.w = live ? gate_decay_fast(b.y + bias_cur.w, gsc, lb, ulb) : 0.0f;
                } else {
                    gv = *reinterpret_cast<const float4 *>(&gs.v[i]);
                }
                acc.x = fmaf(gv.x, kLog2e, acc.x);
                acc.y = fmaf(gv.y, kLog2e, acc.y);
                acc.z = fmaf(gv.z, kLog2e, acc.z);
                acc.w = fmaf(gv.w, kLog2e, acc.w);
                pre[i] = acc;
            }
            *reinterpret_cast<float4 *>(sQS + warp * D + d) = acc;
        }
        if (mbar_wait(full_qk, qkphase)) {
            qkphase ^= 1;
            qkpend = false;
        } else {
            ok = false;
        }
        // 2. row norms of q and k (raw tiles in the A operand's K-major
        //    layout): one (row, 64-channel half) per thread, two threads per row;
        //    step c reads the row's 16-byte unit c ^ (row % 8), so that eight
        //    consecutive rows cover all 32 banks
        {
            const int R = tid >> 1, half = tid & 1;  // R: 0..63 q rows, 64..127 k rows
            const unsigned char *row = sXL + half * 16384 + R * 128;
            float ss = 0.0f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float x[8];
                unpack8(*reinterpret_cast<const uint4 *>(row + ((c ^ (R & 7)) << 4)), x);
#pragma unroll
                for (int t = 0; t < 8; ++t) ss = fmaf(x[t], x[t], ss);
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            if (half == 0) {
                if (R < C) sRq[R] = R < valid ? scale * rsqrtf(ss + 1e-6f) : 0.0f;
                else sRk[R - C] = R - C < valid ? rsqrtf(ss + 1e-6f) : 0.0f;
            }
        }
        // the previous item's W/U staging, under the column operand written
        // next, has been read by its copies
        if (tid == store_tid) bulk_wait_read();
        if (!__syncthreads_and(ok)) {
            ok = false;  // uniform from here on: every thread takes the exit path
            break;
        }

        // 3. per row of the slice, with the reference row m of its half
        //    (m = 15 for rows 0..31, 47 for rows 32..63; log2 units): G_r - G_m,
        //    x = exp(G_r - G_m), and from them the operands q_hat x, k_hat x
        //    (in place over the raw tiles) and the column operand k_hat / x
        //    (hi + lo), so that exp(G_r - G_j) = x_r / x_j for r, j in one half;
        //    rows of the first half also give k_hat e^{G_47 - G_j} = (k_hat / x)
        //    e^{G_47 - G_15} (<= 1), the columns that rows of the second half
        //    pair with them.  E = k_hat x e^{G_m} and QG = q_hat x e^{G_m} (both
        //    k_hat e^{G_r}, q_hat e^{G_r}), KD = (k_hat / x) e^{G_63 - G_m}.  A
        //    chunk with any |G_r - G_m| beyond the limit is deferred as a whole
        //    (its outputs here are discarded: the strong-decay prep rewrites its
        //    record).
        bool wide = false;
        {
            const int hf = warp >> 2;  // this warp's half of the chunk
            float4 before = make_float4(0.f, 0.f, 0.f, 0.f), g15 = before, g47 = before, tot = before;
#pragma unroll
            for (int o = 0; o < 8; ++o) {
                const float4 s = *reinterpret_cast<const float4 *>(sQS + o * D + d);
                if (o < warp) {
                    before.x += s.x; before.y += s.y; before.z += s.z; before.w += s.w;
                }
                if (o < 2) {
                    g15.x += s.x; g15.y += s.y; g15.z += s.z; g15.w += s.w;
                }
                if (o < 6) {
                    g47.x += s.x; g47.y += s.y; g47.z += s.z; g47.w += s.w;
                }
                tot.x += s.x; tot.y += s.y; tot.z += s.z; tot.w += s.w;
            }
            const float4 ref = hf ? g47 : g15;
            const float4 tail = make_float4(tot.x - ref.x, tot.y - ref.y, tot.z - ref.z, tot.w - ref.w);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // pre becomes G_r - G_m
                pre[i].x += before.x - ref.x;
                pre[i].y += before.y - ref.y;
                pre[i].z += before.z - ref.z;
                pre[i].w += before.w - ref.w;
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(pre[i].x), fabsf(pre[i].y)),
                                         fmaxf(fabsf(pre[i].z), fabsf(pre[i].w))));
            }
            wide = !(amax <= kRelLimit2);  // also catches a non-finite decay
            // thread bases: XL (K-major, 128 rows), the column operand (96 rows),
            // 64-row tiles (E, KD), QG rows of WQ
            unsigned char *xl = sXL + kb * 16384 + r0 * 128 + hb;
            unsigned char *cop = sm + P_COL + kb * (2 * NCOL * 128) + r0 * 128 + hb;
            unsigned char *e64 = sE + kb * 8192 + r0 * 128 + hb;
            unsigned char *qg = rec + TcRec::WQ + kb * 16384 + (C + r0) * 128 + hb;
            unsigned char *kd = rec + TcRec::KD + kb * 8192 + r0 * 128 + hb;
            constexpr int kLo = NCOL * 128;  // the lo part's rows follow the hi part's
            // hi + lo bf16 parts of four column values at byte offset `at`
            auto put_col = [&](int at, const float (&c)[4]) {
                const uint2 hi = make_uint2(pack2(c[0], c[1]), pack2(c[2], c[3]));
                const float2 h01 = unpack2(hi.x), h23 = unpack2(hi.y);
                *reinterpret_cast<uint2 *>(cop + at) = hi;
                *reinterpret_cast<uint2 *>(cop + kLo + at) =
                    make_uint2(pack2(c[0] - h01.x, c[1] - h01.y), pack2(c[2] - h23.x, c[3] - h23.y));
            };
            if (hf == 0) {
                // first-half columns again, referenced to row 47, from the raw
                // k tile (before it is overwritten below): k_hat e^{G_47 - G_j},
                // <= 1, its exponent formed directly so that it underflows only
                // where the products it enters are negligible
                const float4 d47 = make_float4(g15.x - g47.x, g15.y - g47.y, g15.z - g47.z, g15.w - g47.w);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int o16 = i * 128 + ((cw ^ i) << 4);
                    const uint2 kraw = *reinterpret_cast<const uint2 *>(xl + 8192 + o16);
                    const bool live = r0 + i < valid;
                    const float2 k01 = unpack2(live ? kraw.x : 0u), k23 = unpack2(live ? kraw.y : 0u);
                    const float rk = sRk[r0 + i];
                    const float c2[4] = {k01.x * rk * ex2(-(pre[i].x + d47.x)), k01.y * rk * ex2(-(pre[i].y + d47.y)),
                                         k23.x * rk * ex2(-(pre[i].z + d47.z)), k23.y * rk * ex2(-(pre[i].w + d47.w))};
                    put_col(o16 + C * 128, c2);
                }
            }
            if (warp == 0)
                *reinterpret_cast<float4 *>(rec + TcRec::GC + 4 * d) =
                    make_float4(ex2(tot.x), ex2(tot.y), ex2(tot.z), ex2(tot.w));
            const float ec[4] = {ex2(ref.x), ex2(ref.y), ex2(ref.z), ex2(ref.w)};
            const float el[4] = {ex2(tail.x), ex2(tail.y), ex2(tail.z), ex2(tail.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int o16 = i * 128 + ((cw ^ i) << 4);  // row r0 + i, this thread's 8 bytes
                const float rel[4] = {pre[i].x, pre[i].y, pre[i].z, pre[i].w};
                const uint2 qraw = *reinterpret_cast<const uint2 *>(xl + o16);
                const uint2 kraw = *reinterpret_cast<const uint2 *>(xl + 8192 + o16);
                const bool live = r0 + i < valid;  // rows past the sequence end: zero
                const float2 q01 = unpack2(live ? qraw.x : 0u), q23 = unpack2(live ? qraw.y : 0u);
                const float2 k01 = unpack2(live ? kraw.x : 0u), k23 = unpack2(live ? kraw.y : 0u);
                const float qv[4] = {q01.x, q01.y, q23.x, q23.y}, kv[4] = {k01.x, k01.y, k23.x, k23.y};
                const float rq = sRq[r0 + i], rk = sRk[r0 + i];
                float qx[4], kx[4], col[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float x = ex2(rel[t]), ir = ex2(-rel[t]);
                    const float kh = kv[t] * rk;
                    qx[t] = qv[t] * rq * x;
                    kx[t] = kh * x;
                    col[t] = kh * ir;
                }
                *reinterpret_cast<uint2 *>(xl + o16) = make_uint2(pack2(qx[0], qx[1]), pack2(qx[2], qx[3]));
                *reinterpret_cast<uint2 *>(xl + 8192 + o16) = make_uint2(pack2(kx[0], kx[1]), pack2(kx[2], kx[3]));
                put_col(o16, col);
                *reinterpret_cast<uint2 *>(e64 + o16) =
                    make_uint2(pack2(kx[0] * ec[0], kx[1] * ec[1]), pack2(kx[2] * ec[2], kx[3] * ec[3]));
                *reinterpret_cast<uint2 *>(qg + o16) =
                    make_uint2(pack2(qx[0] * ec[0], qx[1] * ec[1]), pack2(qx[2] * ec[2], qx[3] * ec[3]));
                *reinterpret_cast<uint2 *>(kd + o16) =
                    make_uint2(pack2(col[0] * el[0], col[1] * el[1]), pack2(col[2] * el[2], col[3] * el[3]));
            }
        }
        // with a scan running alongside (the only reader of the ready flags),
        // the previous item's record is complete once its W/U copies are: its
        // flag goes up here, where warps 4-7 wait for warps 0-3 anyway
        if (scan_ctas && tid == store_tid) {
            bulk_wait_all();
            publish();
        }
        fence_async_smem();
        tc_fence_before();
        const bool defer = __syncthreads_or((int)wide) != 0;
        float beta_nxt = 0.0f, alog_nxt = 0.0f;
        float4 bias_nxt = make_float4(0.f, 0.f, 0.f, 0.f);
        if (defer) {
            // hand the item to the strong-decay prep; the next item's q and k
            // tiles go out at once
            if (tid == 0) {
                defer_list[atomicAdd(defer_count, 1)] = cur.c * H + cur.h;
                atomicOr(status, kStrongDecay);
                load_qk(sm, maps, nxt.h, nxt.tok0, full_qk);
            }
            qkpend = true;
            load_gslice<GATED>(gs, g, gate, nxt.tok0, nxt.valid, r0, nxt.h, H, d);
            if (tid < nxt.valid) beta_nxt = beta_of(nxt.tok0 + tid, nxt.h);
            if (GATED) {
                bias_nxt = *reinterpret_cast<const float4 *>(gate.dt_bias + nxt.h * D + d);
                alog_nxt = gate.a_log[nxt.h];
            }
            if (tid == kPrepThreads - 1 && nxt.valid) *sNext = take_item();
            if (!__syncthreads_and(ok)) {
                ok = false;
                break;
            }
        } else {
        if (tid == 0) {
            tc_fence_after();
            // hi and lo parts side by side in N: TMEM columns 0..95 and 96..191
            mma_tile<128, 2 * NCOL, 128, 128, 2 * NCOL>(tmem, smem_u32(sXL), smem_u32(sm + P_COL), false);
            mma_commit(mbar);
        }
        mpend = true;

        // 4. causal scores A (j <= r, to the record) and the beta-scaled
        //    strictly lower L (to shared fp32 for the inverse): TMEM lanes
        //    0..63 hold A's rows, 64..127 L's; warp w reads the 32 lanes of
        //    quarter w % 4 for output columns j0 = 32 (w / 4) .. +31, which a
        //    row of the first half finds at TMEM columns j (j < 32), a row of
        //    the second half at 64 + j (j < 32) and at j (j >= 32); the lo
        //    part's products sit NCOL columns further and are added.  The v
        //    tile goes out as soon as the column operand has been read.
        float *sL = reinterpret_cast<float *>(sm + P_L);
        if (mbar_wait(mbar, mphase)) {
            mphase ^= 1;
            mpend = false;
        } else {
            ok = false;
        }
        tc_fence_after();
        if (tid == 0 && ok) {
            load_v(sm, maps, cur.h, cur.tok0, full_v);
            vpend = true;
        }
        {
            const int quarter = warp & 3, j0 = 32 * (warp >> 2);
            const bool second = quarter & 1;  // rows 32..63 of A or L
            float x[32];
            if (second || j0 == 0) {
                const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + (second && j0 == 0 ? 64 : j0);
                float xl[32];
                tmem_ld32(ta, x);
                tmem_ld32(ta + NCOL, xl);
                tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 32; ++t) x[t] += xl[t];
            } else {
#pragma unroll
                for (int t = 0; t < 32; ++t) x[t] = 0.0f;  // right of the diagonal
            }
            if (quarter < 2) {
                const int r = 32 * quarter + lane;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] = (j0 + 8 * c8 + t <= r) ? x[8 * c8 + t] : 0.0f;
                    *reinterpret_cast<uint4 *>(rec + TcRec::A + sw128_off(r, j0 + 8 * c8, C)) = pack8(y);
                }
            } else {
                const int r = 32 * (quarter - 2) + lane;
                const float bet = sB[r];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
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
        }
        if (!__syncthreads_and(ok)) {
            ok = false;  // uniform from here on: every thread takes the exit path
            break;
        }

        // 5. X = (I + L)^-1 with L strictly lower (beta-scaled rows), in 16x16
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
        //    Stages B and C hand out (row, 4 columns) slots, 256 at a time.
        {
            const float *cL = sL;
            float *XD = reinterpret_cast<float *>(sm + P_SCR);  // X_aa, a = 0..3
            float *Mb = XD + 4 * MBLK;                         // M_ab, pairs p = 0..5
            float *Cb = reinterpret_cast<float *>(sm + P_L);  // C30, C31 (stage B on: L is consumed)
            float *Xo = Cb + 2 * MBLK;                         // X_10, X_21
            // Block pairs (a, b), a > b, index p: (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
            auto pair_a = [](int p_) { return p_ < 1 ? 1 : (p_ < 3 ? 2 : 3); };
            // T block (a, b), rows i, columns 4c4..4c4+3 from X values x
            auto put_t = [&](int a, int b, int i, int c4, float4 x) {
                const int row = 16 * a + i, col = 16 * b + 4 * c4;
                const float4 bt = *reinterpret_cast<const float4 *>(sB + col);
                const float y0 = x.x * bt.x, y1 = x.y * bt.y, y2 = x.z * bt.z, y3 = x.w * bt.w;
                const uint32_t h01 = pack2(y0, y1), h23 = pack2(y2, y3);
                const float2 f01 = unpack2(h01), f23 = unpack2(h23);
                const uint32_t off = sw128_off(row, col, 64);
                const uint2 hi = make_uint2(h01, h23);
                const uint2 lo = make_uint2(pack2(y0 - f01.x, y1 - f01.y), pack2(y2 - f23.x, y3 - f23.y));
                // rows 64..127 repeat rows 0..63, so that W and U land in both
                // halves of TMEM and all eight warps share their readout
                *reinterpret_cast<uint2 *>(sT + off) = hi;
                *reinterpret_cast<uint2 *>(sT + 8192 + off) = hi;
                *reinterpret_cast<uint2 *>(sT + 16384 + off) = lo;
                *reinterpret_cast<uint2 *>(sT + 24576 + off) = lo;
            };
            if (warp < 5) {
                const int sl = 32 * warp + lane;
                const bool unit = sl < 64;
                const int p_ = unit ? 0 : (sl - 64) >> 4;
                const int a = unit ? sl >> 4 : pair_a(p_);
                const int b = unit ? a : p_ - a * (a - 1) / 2;
                const int c = sl & 15, o = 16 * a;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float lr[16];
                    row16(cL + o, LSTRIDE, o + r, lr);
                    const float rhs = unit ? (r == c ? 1.0f : 0.0f) : cL[(o + r) * LSTRIDE + 16 * b + c];
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
            } else {
                // meanwhile warps 5-7: zeros above the block diagonal of T, 6
                // blocks x 16 rows x 2 chunks x hi, lo (4 slots per thread)
                for (int sl = tid - 160; sl < 384; sl += 96) {
                    const int pz = sl >> 6, i = (sl >> 2) & 15, h = (sl >> 1) & 1, hl = sl & 1;
                    const int a = pz < 3 ? 0 : (pz < 5 ? 1 : 2);
                    const int b = pz < 3 ? pz + 1 : (pz < 5 ? pz - 1 : 3);
                    unsigned char *z = sT + hl * 16384 + sw128_off(16 * a + i, 16 * b + 8 * h, 64);
                    *reinterpret_cast<uint4 *>(z) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(z + 8192) = make_uint4(0, 0, 0, 0);
                }
                // and the item after next, claimed here, where these warps wait
                // for the substitutions anyway (the later an item is claimed,
                // the less the CTAs' ends spread when the items run out);
                // handed over in shared memory
                if (tid == kPrepThreads - 1 && nxt.valid) *sNext = take_item();
            }
            __syncthreads();
            if (tid < 192) {  // X_{q+1,q} = -M_{q+1,q} X_qq, one (row, 4 columns) slot per thread
                const int ii = (tid >> 2) & 15, c4 = tid & 3, q_ = tid >> 6;
                const int pm = q_ == 0 ? 0 : (q_ == 1 ? 2 : 5);
                float4 x = mm16_row4(Mb + pm * MBLK, MS, XD + q_ * MBLK, MS, ii, c4);
                x = make_float4(-x.x, -x.y, -x.z, -x.w);
                if (q_ < 2) *reinterpret_cast<float4 *>(Xo + q_ * MBLK + ii * MS + 4 * c4) = x;
                put_t(q_ + 1, q_, ii, c4, x);
            } else {  // C30 = M_32 M_20 - M_30, C31 = M_32 M_21 - M_31: two slots per thread
#pragma unroll 1
                for (int k_ = 0; k_ < 2; ++k_) {
                    const int sl = tid - 192, ii = (sl >> 2) & 15, c4 = sl & 3;
                    float4 x = mm16_row4(Mb + 5 * MBLK, MS, Mb + (k_ == 0 ? 1 : 2) * MBLK, MS, ii, c4);
                    const float4 m = *reinterpret_cast<const float4 *>(Mb + (3 + k_) * MBLK + ii * MS + 4 * c4);
                    *reinterpret_cast<float4 *>(Cb + k_ * MBLK + ii * MS + 4 * c4) =
                        make_float4(x.x - m.x, x.y - m.y, x.z - m.z, x.w - m.w);
                }
            }
            __syncthreads();
            if (tid < 192) {
                const int q_ = tid >> 6, ii = (tid >> 2) & 15, c4 = tid & 3;
                float a16[16];
                float4 x, y;
                if (q_ == 0) {         // X_20 = -(M_20 X_00 + M_21 X_10)
                    row16(Mb + 1 * MBLK, MS, ii, a16);
                    x = row4_times(a16, XD, c4);
                    row16(Mb + 2 * MBLK, MS, ii, a16);
                    y = row4_times(a16, Xo, c4);
                    put_t(2, 0, ii, c4, make_float4(-(x.x + y.x), -(x.y + y.y), -(x.z + y.z), -(x.w + y.w)));
                } else if (q_ == 1) {  // X_31 = -(M_31 X_11 + M_32 X_21)
                    row16(Mb + 4 * MBLK, MS, ii, a16);
                    x = row4_times(a16, XD + MBLK, c4);
                    row16(Mb + 5 * MBLK, MS, ii, a16);
                    y = row4_times(a16, Xo + MBLK, c4);
                    put_t(3, 1, ii, c4, make_float4(-(x.x + y.x), -(x.y + y.y), -(x.z + y.z), -(x.w + y.w)));
                } else {               // X_30 = C30 X_00 + C31 X_10
                    row16(Cb, MS, ii, a16);
                    x = row4_times(a16, XD, c4);
                    row16(Cb + MBLK, MS, ii, a16);
                    y = row4_times(a16, Xo, c4);
                    put_t(3, 0, ii, c4, make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w));
                }
            } else {  // the diagonal blocks of T: 4 blocks x 16 rows x 4 column groups, 4 per thread
#pragma unroll 1
                for (int k_ = 0; k_ < 4; ++k_) {
                    const int sl = tid - 192 + 64 * k_;
                    const int a = sl >> 6, ii = (sl >> 2) & 15, c4 = sl & 3;
                    put_t(a, a, ii, c4, *reinterpret_cast<const float4 *>(XD + a * MBLK + ii * MS + 4 * c4));
                }
            }
        }
        // the v tile (requested after the A/L MMA): rows past the sequence
        // end are zeroed
        if (mbar_wait(full_v, vphase)) {
            vphase ^= 1;
            vpend = false;
        } else {
            ok = false;
        }
        for (int i = tid; i < (C - valid) * 16; i += kPrepThreads) {
            const int r = valid + i / 16, c16 = i % 16;
            *reinterpret_cast<uint4 *>(sm + P_V + (c16 >> 3) * 8192 + r * 128 + (c16 & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) {
            ok = false;  // uniform from here on: every thread takes the exit path
            break;
        }
        // 6. W = T E, U = T V (hi + lo T); the q and k tiles of the next item
        //    go out now (L and the inverse scratch are consumed), and its g
        //    slice and beta are fetched into registers while the MMA runs.
        if (tid == 0) {
            tc_fence_after();
            // [U | W] = T [v | E]: one N = 256 group (TMEM columns 0..127 U, 128..255 W)
            mma_tile<128, 256, 64, 128, 64, false, true>(tmem, smem_u32(sT), smem_u32(sm + P_V), false);
            mma_tile<128, 256, 64, 128, 64, false, true>(tmem, smem_u32(sT + 16384), smem_u32(sm + P_V), true);
            mma_commit(mbar);
            load_qk(sm, maps, nxt.h, nxt.tok0, full_qk);
        }
        mpend = true;
        qkpend = true;
        load_gslice<GATED>(gs, g, gate, nxt.tok0, nxt.valid, r0, nxt.h, H, d);
        if (tid < nxt.valid) beta_nxt = beta_of(nxt.tok0 + tid, nxt.h);
        if (GATED) {
            bias_nxt = *reinterpret_cast<const float4 *>(gate.dt_bias + nxt.h * D + d);
            alog_nxt = gate.a_log[nxt.h];
        }
        if (mbar_wait(mbar, mphase)) {
            mphase ^= 1;
            mpend = false;
        } else {
            ok = false;
        }
        tc_fence_after();

        // 7. W and U rows (TMEM lanes 0..63, repeated in lanes 64..127): warp
        //    w reads lane quarter w % 4, i.e. rows 32 (w % 2) .. +31, columns
        //    64 ((w % 4) / 2) .. +63 of W (w < 4) or U (w >= 4) -> shared
        //    memory in the record's own layout -> three bulk copies to the
        //    record.  U rows are stored with their 16-byte chunks rotated
        //    (chunk c of row i at c ^ ((i / 2) % 4)), which keeps these writes
        //    and the scan's reads free of bank conflicts.
        unsigned char *stg = sm + P_STAGE;
        {
            const int quarter = warp & 3, part = warp >> 2;
            const int i = 32 * (quarter & 1) + lane, c0 = 64 * (quarter >> 1);
            const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + 128 * (1 - part) + c0;
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                float x[32];
                tmem_ld32(ta + 32 * cb, x);
                tmem_ld_wait();
                const int col = c0 + 32 * cb;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t];
                    unsigned char *dst = part == 0
                        ? stg + sw128_off(i, col + 8 * c8, 64)
                        : stg + 16384 + (col >> 5) * TcRec::UBLK + i * 64 + ((c8 ^ ((i >> 1) & 3)) << 4);
                    *reinterpret_cast<uint4 *>(dst) = pack8(y);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) {
            ok = false;  // uniform from here on: every thread takes the exit path
            break;
        }
        if (tid == store_tid) {
            bulk_s2g(rec + TcRec::WQ, stg, 8192);                  // W, key columns 0..63
            bulk_s2g(rec + TcRec::WQ + 16384, stg + 8192, 8192);   // W, key columns 64..127
            bulk_s2g(rec + TcRec::U, stg + 16384, 4 * TcRec::UBLK);
            bulk_commit();
            *sPub = cur.c * H + cur.h;
        }
        }
        if (!nxt.valid) break;
        cur = nxt;
        nxt = *sNext;
        beta_cur = beta_nxt;
        bias_cur = bias_nxt;
        alog_cur = alog_nxt;
    }
    if (tid == store_tid) {
        bulk_wait_all();  // the last record's W and U are written
        publish();
    }
    if (tid == 0) {
        // the tiles requested for the item of no rows after the last one (or,
        // on the exit path, whatever copies and MMAs are still in flight) land
        // before the shared memory and the TMEM are released
        if (qkpend) mbar_wait(full_qk, qkphase, 400000000LL);
        if (!ok) {
            atomicOr(status, kStatusTimeout);
            if (vpend) mbar_wait(full_v, vphase, 400000000LL);
            if (mpend) mbar_wait(mbar, mphase, 400000000LL);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
    if (tid == 0) count_release(prep_done);
}

// ---------------------------------------------------------------------------
// scan
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 160;  // warps 0-3: state rows, Vn, output rows; warp 4: MMAs and loads
constexpr int kIssuer = 128;       // lane 0 of warp 4
constexpr int kSplitThreads = 192;  // the split scan: warp 5 issues the second key half of D1
constexpr int kIssuer2 = 160;       // lane 0 of warp 5
constexpr uint32_t kSplitTmemCols = 256;  // D1 (2 buffers x 2 key halves x 32 columns), D3 (32)
constexpr int BV = 32;
constexpr int kStages = 3;
static_assert(BV == 32, "S and Vn are N = 32 operands");
constexpr uint32_t kImageBytes = TcRec::U;                   // WQ | KD | A | gC
constexpr uint32_t kStageBytes = kImageBytes + TcRec::UBLK;  // + this CTA's U block
constexpr int S_STAGE = 62464;                               // kStageBytes rounded up to 1024
constexpr int S_SOP = kStages * S_STAGE;                     // S operand [128 keys][32] bf16, 8 KB
constexpr int S_VOP = S_SOP + 8192;                          // Vn operand [64 rows][32] bf16, 4 KB
constexpr int S_BAR = S_VOP + 4096;                          // mbarriers, tmem slot
constexpr int S_BYTES = S_BAR + 128;
constexpr int S_SMEM = S_BYTES + 1024;
static_assert(kStageBytes <= (uint32_t)S_STAGE, "stage too small");
static_assert(kImageBytes % 16 == 0 && TcRec::UBLK % 16 == 0, "bulk copy size");
static_assert(8 * (kStages + 4) + 4 <= 128, "scan barrier block");
// named barriers: S operand ready (every warp), Vn ready (warps 0-4: the Vn
// warps, the issuer, and the output warps once they have stored the previous
// chunk's rows)
constexpr uint32_t kBarS = 1, kBarV = 2;

// The split scan's shared memory: two "front" slots (the part a chunk step
// needs first: WQ for D1, U for Vn, gC for the state update) and one KD | A
// slot (read only by the step's last two MMAs), so that a CTA fits beside a
// prep CTA on one SM and runs alongside the prep.
constexpr uint32_t kFBytes = 32768 + 512 + TcRec::UBLK;  // WQ | gC | this CTA's U block
constexpr uint32_t kKBytes = TcRec::GC - TcRec::KD;     // KD | A, contiguous in the record
constexpr int SP_F = 37888;                             // front slot (kFBytes rounded up to 1024)
constexpr int SP_FGC = 32768;                           // gC in a front slot
constexpr int SP_FU = SP_FGC + 512;                     // U block in a front slot
constexpr int SP_K = 2 * SP_F;                          // KD | A slot, 24 KB
constexpr int SP_SOP = SP_K + 24576;                    // S operand [128 keys][32] bf16, 8 KB
constexpr int SP_VOP = SP_SOP + 8192;                   // Vn operand [64 rows][32] bf16, 4 KB
constexpr int SP_BAR = SP_VOP + 4096;                   // mbarriers, tmem slot
constexpr int SP_BYTES = SP_BAR + 128;
// more than half of an SM's 228 KB (with the 1 KB each CTA reserves), so that
// the scan's CTAs spread one per SM, and room for one prep CTA beside each
constexpr int SP_SMEM = 116736;
static_assert(kFBytes <= (uint32_t)SP_F && TcRec::A - TcRec::KD == 16384 && kKBytes == 24576,
              "split scan slots");
static_assert(SP_BYTES + 1024 <= SP_SMEM && 2 * (SP_SMEM + 1024) > 233472 &&
                  SP_SMEM + 1024 + P_SMEM + 1024 <= 233472,
              "one split-scan CTA per SM, beside one prep CTA");
static_assert(8 * 7 + 4 <= 128, "split scan barrier block");

// This thread's 32 values x[v] as row k of an N = 32 operand (MN-major,
// 64-byte swizzle, see sw64_off): four 16-byte stores, conflict-free across
// a warp of consecutive rows.
__device__ __forceinline__ void store_row_n32(unsigned char *op, int k, const float (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float y[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) y[t] = x[8 * c + t];
        *reinterpret_cast<uint4 *>(op + sw64_off(k, 8 * c)) = pack8(y);
    }
}

// Per chunk ck (records staged by bulk copies, kStages deep), D1 = D1[ck & 1]:
//   issuers:    D1 = [W ; QG] S, keys 0..63 from warp 4 and keys 64..127 from
//               warp 5 into two accumulators              after "S ready"
//   warps 0-1:  Vn = U - (D1a + D1b)[0:64] -> Vn operand  -> "Vn ready"
//   warps 2-3:  output rows of chunk ck-1 from D1[(ck-1) & 1]
//   issuer:     D3 = KD^T Vn, then D1a[64:128] += A Vn    after "Vn ready"
//   warps 0-3:  S = diag(gC) S + D3 -> S operand          -> "S ready"
// Dedicated issuing warps keep the (slow to issue) MMAs off the threads that
// own state rows; a tcgen05.mma costs its issuing thread ~60 cycles, so D1's
// eight instructions go out as two groups of four at once (scan 76 -> 74 us
// on the 4k workload).  The output MMA runs while the state is updated.
__global__ void __launch_bounds__(kSplitThreads, 1)
    chunk_scan_tc_kernel(const float *__restrict__ initial_state, float *__restrict__ final_state,
                         const int32_t *__restrict__ state_indices, __nv_bfloat16 *__restrict__ o,
                         int n_seqs, int H, void *workspace, WsLayout L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sS = sm + S_SOP;
    unsigned char *sVn = sm + S_VOP;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + S_BAR);
    uint64_t *bar_ws = full + kStages;  // D1 = WQ S done
    uint64_t *bar_d3 = bar_ws + 1;      // D3 = KD^T Vn done
    uint64_t *bar_out = bar_d3 + 1;     // D1 += A Vn done: the chunk's output rows
    uint64_t *bar_drain = bar_out + 1;  // exit path: every MMA issued so far is done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_drain + 1);
    griddep_wait();  // the records (previous kernel) are complete
    // the next forward's chunk index may be scheduled (one CTA; it waits for
    // this grid to complete before it writes anything)
    griddep_launch_dependents();

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
    auto stage_of = [&](int ck) { return sm + (ck % kStages) * S_STAGE; };
    auto issue = [&](int ck) {  // the issuing thread
        unsigned char *dst = stage_of(ck);
        uint64_t *b = &full[ck % kStages];
        mbar_arrive_expect_tx(b, kStageBytes);
        bulk_g2s(dst, rec_of(ck), kImageBytes, b);
        bulk_g2s(dst + kImageBytes, rec_of(ck) + TcRec::U + vb * TcRec::UBLK, TcRec::UBLK, b);
    };

    if (warp == 0) tmem_alloc(tmem_slot, kSplitTmemCols);
    if (tid == kIssuer) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        mbar_init(bar_ws, 2);  // both key halves of D1
        mbar_init(bar_d3, 1);
        mbar_init(bar_out, 1);
        mbar_init(bar_drain, 2);  // both issuers
        fence_mbar_init();
    }
    // state row d = tid (warps 0-3), columns v0 .. v0+31, fp32 in registers
    float S[BV];
    if (tid < D) {
#pragma unroll
        for (int x = 0; x < BV; ++x)
            S[x] = initial_state ? initial_state[st_off + (int64_t)(v0 + x) * D + tid] : 0.0f;
        store_row_n32(sS, tid, S);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tD3 = tmem + 128;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

    // Output rows of chunk ck (TMEM D1 buffer ck & 1, both key halves, lanes 64..127) -> o
    // (warps 2-3).
    auto store_output = [&](int ck) {
        float x[32], x2[32];
        tmem_ld32(tmem + 32 * (ck & 1) + lane_base, x);
        tmem_ld32(tmem + 64 + 32 * (ck & 1) + lane_base, x2);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 32; ++t) x[t] += x2[t];
        const int r = tid - 64;
        if (r < min(C, len - ck * C)) {
            const int64_t tok = (int64_t)start + (int64_t)ck * C + r;
            uint4 *op = reinterpret_cast<uint4 *>(o + (tok * H + h) * (int64_t)D + v0);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float y[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t];
                op[c8] = pack8(y);
            }
        }
    };

    // stage loads issued / waited for by the issuer, for the exit path
    int loads_issued = 0, loads_done = 0;
    if (tid == kIssuer)
        for (int ck = 0; ck < kStages - 1 && ck < nck; ++ck, ++loads_issued) issue(ck);
    bool ok = true;
    for (int ck = 0; ck < nck; ++ck) {
        const uint32_t fpar = (uint32_t)((ck / kStages) & 1), cpar = (uint32_t)(ck & 1);
        unsigned char *st = stage_of(ck);
        const uint32_t tD1 = tmem + 32 * (ck & 1);
        if (tid == kIssuer) {
            ok = mbar_wait(&full[ck % kStages], fpar) && ok;
            if (ok) loads_done = ck + 1;
            tc_fence_after();
            if (ok) {  // keys 0..63 of D1 = [W ; QG] S
                mma_tile_n32<128, 64, 128>(tD1, smem_u32(st + TcRec::WQ), smem_u32(sS), false);
                mma_commit(bar_ws);
            }
            // refill the stage of chunk ck-1 once its last MMA (D1 += A Vn) is done
            const int t = ck + kStages - 1;
            if (ok && t < nck) {
                if (ck > 0) ok = mbar_wait(bar_out, cpar ^ 1) && ok;
                if (ok) {
                    issue(t);
                    ++loads_issued;
                }
            }
        } else if (tid == kIssuer2) {
            ok = mbar_wait(&full[ck % kStages], fpar) && ok;
            tc_fence_after();
            if (ok) {  // keys 64..127 of D1, issued at the same time from a second thread
                mma_tile_n32<128, 64, 128>(tD1 + 64, smem_u32(st + TcRec::WQ + 16384), smem_u32(sS + 4096),
                                           false);
                mma_commit(bar_ws);
            }
        } else if (warp < 2) {
            ok = mbar_wait(&full[ck % kStages], fpar) && ok;  // U of this stage
            float x[32], x2[32], u[32];  // Vn = U - W S, row tid
            {  // U first, while D1 is formed
                const uint4 *up = reinterpret_cast<const uint4 *>(st + kImageBytes + tid * 64);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
                    unpack8(up[c8 ^ ((tid >> 1) & 3)], y);
#pragma unroll
                    for (int t = 0; t < 8; ++t) u[8 * c8 + t] = y[t];
                }
            }
            ok = mbar_wait(bar_ws, cpar) && ok;
            tc_fence_after();
            tmem_ld32(tD1 + lane_base, x);
            tmem_ld32(tD1 + 64 + lane_base, x2);
            tmem_ld_wait();
#pragma unroll
            for (int vv = 0; vv < BV; ++vv) x[vv] = u[vv] - (x[vv] + x2[vv]);
            store_row_n32(sVn, tid, x);
            fence_async_smem();
            tc_fence_before();
        } else if (warp < 4) {
            ok = mbar_wait(&full[ck % kStages], fpar) && ok;  // gC of this stage
            if (ck > 0) {
                ok = mbar_wait(bar_out, cpar ^ 1) && ok;
                tc_fence_after();
                if (ok) store_output(ck - 1);
            }
            tc_fence_before();
        }
        // (a failure seen here is carried to the "S ready" barrier below, which
        // every warp reaches.)  The output warps meet "Vn ready" too: they wait
        // on bar_out's phase of chunk ck-1 by parity, so the issuer must not
        // complete chunk ck's phase (D1 += A Vn, issued after this barrier)
        // before they have seen the previous one.
        if (warp < 5) ok = named_bar_and(kBarV, 160, ok);
        if (tid == kIssuer) {
            tc_fence_after();
            if (ok) {
                mma_tile_n32<128, 64, 64, true>(tD3, smem_u32(st + TcRec::KD), smem_u32(sVn), false);
                mma_commit(bar_d3);
                mma_tile_n32<128, 64, 128>(tD1, smem_u32(st + TcRec::A) - 8192, smem_u32(sVn), true);
                mma_commit(bar_out);
            }
        } else if (warp < 4 && ok) {
            const float gc = reinterpret_cast<const float *>(st + TcRec::GC)[tid];
            ok = mbar_wait(bar_d3, cpar) && ok;
            tc_fence_after();
            float x[32];  // S = diag(gC) S + KD^T Vn
            tmem_ld32(tD3 + lane_base, x);
            tmem_ld_wait();
#pragma unroll
            for (int vv = 0; vv < BV; ++vv) S[vv] = fmaf(gc, S[vv], x[vv]);
            store_row_n32(sS, tid, S);
            fence_async_smem();
            tc_fence_before();
        }
        if (!named_bar_and(kBarS, kSplitThreads, ok)) {
            ok = false;
            break;
        }
    }
    if (ok && nck > 0 && (warp == 2 || warp == 3)) {
        ok = mbar_wait(bar_out, (uint32_t)((nck - 1) & 1));
        tc_fence_after();
        if (ok) store_output(nck - 1);
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        // let copies and MMAs still in flight land before the shared memory
        // and the TMEM are released
        if (tid == kIssuer2) mma_commit(bar_drain);
        if (tid == kIssuer) {
            atomicOr(status, kStatusTimeout);
            for (int t = loads_done; t < loads_issued; ++t)
                mbar_wait(&full[t % kStages], (uint32_t)((t / kStages) & 1), 400000000LL);
            mma_commit(bar_drain);
            mbar_wait(bar_drain, 0, 400000000LL);
        }
    } else if (final_state && tid < D) {
#pragma unroll
        for (int x = 0; x < BV; ++x) final_state[st_off + (int64_t)(v0 + x) * D + tid] = S[x];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kSplitTmemCols);
}

// Per chunk ck, D1 = D1[ck & 1]:
//   issuers:    D1 = [W ; QG] S, keys 0..63 from warp 4 and keys 64..127 from
//               warp 5 into two accumulators              after "S ready"
//   warps 0-1:  Vn = U - (D1a + D1b)[0:64] -> Vn operand  -> "Vn ready"
//   warps 2-3:  output rows of chunk ck-1 from D1[(ck-1) & 1]
//   issuer:     D3 = KD^T Vn, then D1a[64:128] += A Vn    after "Vn ready"
//   warps 0-3:  S = diag(gC) S + D3 -> S operand          -> "S ready"
// Dedicated issuing warps keep the (slow to issue) MMAs off the threads that
// own state rows; a tcgen05.mma costs its issuing thread ~60 cycles, so D1's
// eight instructions go out as two groups of four at once.  The output MMA
// runs while the state is updated.
// Loads (all from the issuer): the front part of chunk ck+1 (WQ, gC, U) right
// after D1 of chunk ck, into the front slot chunk ck-1 used; its KD | A once
// D1 += A Vn of chunk ck has read the single KD | A slot.  Each waits for the
// record's ready flag, so the scan can run alongside the prep that writes the
// records (launched after it); with the records already written the flags
// are up.  Registers are capped at 128 per thread (TMEM read in 16-column
// halves where three 32-column rows would be live): an SM sub-partition holds
// 16 K registers, and a scan CTA (6 warps, two on each of two sub-partitions)
// shares its SM with a prep CTA (8 warps of 128 registers, two per
// sub-partition).
__global__ void __maxnreg__(128)
    chunk_scan_tc_overlap_kernel(const float *__restrict__ initial_state, float *__restrict__ final_state,
                         const int32_t *__restrict__ state_indices, __nv_bfloat16 *__restrict__ o,
                         int n_seqs, int H, void *workspace, WsLayout L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sK = sm + SP_K;
    unsigned char *sS = sm + SP_SOP;
    unsigned char *sVn = sm + SP_VOP;
    uint64_t *full_f = reinterpret_cast<uint64_t *>(sm + SP_BAR);  // front slots 0, 1
    uint64_t *full_k = full_f + 2;      // the KD | A slot
    uint64_t *bar_ws = full_k + 1;      // D1 = WQ S done
    uint64_t *bar_d3 = bar_ws + 1;      // D3 = KD^T Vn done
    uint64_t *bar_out = bar_d3 + 1;     // D1 += A Vn done: the chunk's output rows
    uint64_t *bar_drain = bar_out + 1;  // exit path: every MMA issued so far is done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_drain + 1);
    griddep_wait();  // the chunk index (and, launched after the prep, the records) is complete
    // the next kernel may be scheduled: the prep, when it runs alongside (it
    // waits for no part of this grid), or the next forward's chunk index (one
    // CTA, which waits for this grid to complete before it writes anything)
    griddep_launch_dependents();

    const int n = blockIdx.x, h = blockIdx.y, vb = blockIdx.z, v0 = vb * BV;
    const int tid = threadIdx.x, warp = tid >> 5;
    int32_t *scan_done = ws_at<int32_t>(workspace, L.scan_done_off);
    const int32_t start = ws_at<const int32_t>(workspace, L.seq_start_off)[n];
    if (start < 0) {  // sequence skipped (bad cu_seqlens or slot)
        if (tid == 0) count_release(scan_done);
        return;
    }
    const int len = ws_at<const int32_t>(workspace, L.seq_len_off)[n];
    const int c0 = ws_at<const int32_t>(workspace, L.chunk_off_off)[n];
    const int nck = (len + C - 1) / C;
    const int64_t slot = state_indices ? (int64_t)state_indices[n] : (int64_t)n;
    const int64_t st_off = (slot * H + h) * (int64_t)D * D;  // [V][K] block of (slot, h)
    int32_t *status = ws_at<int32_t>(workspace, L.status_off);
    const unsigned char *recs = ws_at<const unsigned char>(workspace, L.records_off);
    const int32_t *ready = ws_at<const int32_t>(workspace, L.ready_off);
    auto rec_of = [&](int ck) { return recs + ((size_t)(c0 + ck) * H + h) * TcRec::bytes; };
    auto flag_of = [&](int ck) { return ready + (size_t)(c0 + ck) * H + h; };
    auto fslot = [&](int ck) { return sm + (ck & 1) * SP_F; };
    auto issue_f = [&](int ck) {  // the issuer, after the record's flag
        unsigned char *dst = fslot(ck);
        uint64_t *b = &full_f[ck & 1];
        const unsigned char *r = rec_of(ck);
        mbar_arrive_expect_tx(b, kFBytes);
        bulk_g2s(dst, r + TcRec::WQ, 32768, b);
        bulk_g2s(dst + SP_FGC, r + TcRec::GC, 512, b);
        bulk_g2s(dst + SP_FU, r + TcRec::U + vb * TcRec::UBLK, TcRec::UBLK, b);
    };
    auto issue_k = [&](int ck) {  // the issuer, after the record's flag
        mbar_arrive_expect_tx(full_k, kKBytes);
        bulk_g2s(sK, rec_of(ck) + TcRec::KD, kKBytes, full_k);
    };

    if (warp == 0) tmem_alloc(tmem_slot, kSplitTmemCols);
    if (tid == kIssuer) {
        mbar_init(&full_f[0], 1);
        mbar_init(&full_f[1], 1);
        mbar_init(full_k, 1);
        mbar_init(bar_ws, 2);  // both key halves of D1
        mbar_init(bar_d3, 1);
        mbar_init(bar_out, 1);
        mbar_init(bar_drain, 2);  // both issuers
        fence_mbar_init();
    }
    // state row d = tid (warps 0-3), columns v0 .. v0+31, fp32 in registers
    float S[BV];
    if (tid < D) {
#pragma unroll
        for (int x = 0; x < BV; ++x)
            S[x] = initial_state ? initial_state[st_off + (int64_t)(v0 + x) * D + tid] : 0.0f;
        store_row_n32(sS, tid, S);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tD3 = tmem + 128;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

    // Output rows of chunk ck (TMEM D1 buffer ck & 1, both key halves, lanes 64..127) -> o
    // (warps 2-3), 16 columns at a time.
    auto store_output = [&](int ck) {
        const int r = tid - 64;
        const bool live = r < min(C, len - ck * C);
        uint4 *op = reinterpret_cast<uint4 *>(o + (((int64_t)start + (int64_t)ck * C + r) * H + h) * (int64_t)D + v0);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float x[16], x2[16];
            tmem_ld16(tmem + 32 * (ck & 1) + 16 * hf + lane_base, x);
            tmem_ld16(tmem + 64 + 32 * (ck & 1) + 16 * hf + lane_base, x2);
            tmem_ld_wait();
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {
                float y[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t] + x2[8 * c8 + t];
                if (live) op[2 * hf + c8] = pack8(y);
            }
        }
    };

    // loads issued / waited for, for the exit path (all from the issuer)
    int f_issued = 0, f_done = 0, k_issued = 0;
    bool ok = true;
    if (nck > 0 && tid == kIssuer) {
        ok = flag_wait(flag_of(0));
        if (ok) {
            issue_f(0);
            issue_k(0);
            f_issued = 1;
            k_issued = 1;
        }
    }
    for (int ck = 0; ck < nck; ++ck) {
        const uint32_t fpar = (uint32_t)((ck >> 1) & 1), cpar = (uint32_t)(ck & 1);
        unsigned char *fs = fslot(ck);
        const uint32_t tD1 = tmem + 32 * (ck & 1);
        const bool more = ck + 1 < nck;
        if (tid == kIssuer) {
            ok = mbar_wait(&full_f[ck & 1], fpar) && ok;
            if (ok) f_done = ck + 1;
            tc_fence_after();
            if (ok) {  // keys 0..63 of D1 = [W ; QG] S
                mma_tile_n32<128, 64, 128>(tD1, smem_u32(fs), smem_u32(sS), false);
                mma_commit(bar_ws);
            }
            // the next chunk's front part, into the slot of chunk ck-1 (whose
            // readers have all passed "S ready" of chunk ck-1)
            if (ok && more) {
                ok = flag_wait(flag_of(ck + 1));
                if (ok) {
                    issue_f(ck + 1);
                    ++f_issued;
                }
            }
        } else if (tid == kIssuer2) {
            ok = mbar_wait(&full_f[ck & 1], fpar) && ok;
            tc_fence_after();
            if (ok) {  // keys 64..127 of D1, issued at the same time from a second thread
                mma_tile_n32<128, 64, 128>(tD1 + 64, smem_u32(fs + 16384), smem_u32(sS + 4096), false);
                mma_commit(bar_ws);
            }
        } else if (warp < 2) {
            ok = mbar_wait(&full_f[ck & 1], fpar) && ok;  // U of this chunk
            uint4 up[4];  // U row tid (bf16), read while D1 is formed
            {
                const uint4 *ur = reinterpret_cast<const uint4 *>(fs + SP_FU + tid * 64);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) up[c8] = ur[c8 ^ ((tid >> 1) & 3)];
            }
            ok = mbar_wait(bar_ws, cpar) && ok;
            tc_fence_after();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {  // Vn = U - W S, row tid, 16 columns at a time
                float x[16], x2[16];
                tmem_ld16(tD1 + 16 * hf + lane_base, x);
                tmem_ld16(tD1 + 64 + 16 * hf + lane_base, x2);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float y[8];
                    unpack8(up[2 * hf + c], y);
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] -= x[8 * c + t] + x2[8 * c + t];
                    *reinterpret_cast<uint4 *>(sVn + sw64_off(tid, 16 * hf + 8 * c)) = pack8(y);
                }
            }
            fence_async_smem();
            tc_fence_before();
        } else if (warp < 4) {
            ok = mbar_wait(&full_f[ck & 1], fpar) && ok;  // gC of this chunk
            if (ck > 0) {
                ok = mbar_wait(bar_out, cpar ^ 1) && ok;
                tc_fence_after();
                if (ok) store_output(ck - 1);
            }
            tc_fence_before();
        }
        // (a failure seen here is carried to the "S ready" barrier below, which
        // every warp reaches.)  The output warps meet "Vn ready" too: they wait
        // on bar_out's phase of chunk ck-1 by parity, so the issuer must not
        // complete chunk ck's phase (D1 += A Vn, issued after this barrier)
        // before they have seen the previous one.
        if (warp < 5) ok = named_bar_and(kBarV, 160, ok);
        if (tid == kIssuer) {
            if (ok) ok = mbar_wait(full_k, cpar);  // KD | A of this chunk
            tc_fence_after();
            if (ok) {
                mma_tile_n32<128, 64, 64, true>(tD3, smem_u32(sK), smem_u32(sVn), false);
                mma_commit(bar_d3);
                mma_tile_n32<128, 64, 128>(tD1, smem_u32(sK + 16384) - 8192, smem_u32(sVn), true);
                mma_commit(bar_out);
            }
            // the next chunk's KD | A (its flag seen above), once this chunk's
            // last MMA has read the slot
            if (ok && more) {
                ok = mbar_wait(bar_out, cpar);
                if (ok) {
                    issue_k(ck + 1);
                    ++k_issued;
                }
            }
        } else if (warp < 4 && ok) {
            const float gc = reinterpret_cast<const float *>(fs + SP_FGC)[tid];
            ok = mbar_wait(bar_d3, cpar) && ok;
            tc_fence_after();
            float x[32];  // S = diag(gC) S + KD^T Vn
            tmem_ld32(tD3 + lane_base, x);
            tmem_ld_wait();
#pragma unroll
            for (int vv = 0; vv < BV; ++vv) S[vv] = fmaf(gc, S[vv], x[vv]);
            store_row_n32(sS, tid, S);
            fence_async_smem();
            tc_fence_before();
        }
        if (!named_bar_and(kBarS, kSplitThreads, ok)) {
            ok = false;
            break;
        }
    }
    if (ok && nck > 0 && (warp == 2 || warp == 3)) {
        ok = mbar_wait(bar_out, (uint32_t)((nck - 1) & 1));
        tc_fence_after();
        if (ok) store_output(nck - 1);
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        // let copies and MMAs still in flight land before the shared memory
        // and the TMEM are released (at most one KD | A copy is in flight: a
        // new one goes out only after the previous one was consumed)
        if (tid == kIssuer2) mma_commit(bar_drain);
        if (tid == kIssuer) {
            atomicOr(status, kStatusTimeout);
            for (int t = f_done; t < f_issued; ++t)
                mbar_wait(&full_f[t & 1], (uint32_t)((t >> 1) & 1), 400000000LL);
            if (k_issued > 0) mbar_wait(full_k, (uint32_t)((k_issued - 1) & 1), 400000000LL);
            mma_commit(bar_drain);
            mbar_wait(bar_drain, 0, 400000000LL);
        }
    } else if (final_state && tid < D) {
#pragma unroll
        for (int x = 0; x < BV; ++x) final_state[st_off + (int64_t)(v0 + x) * D + tid] = S[x];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kSplitTmemCols);
    if (tid == 0) count_release(scan_done);  // this CTA's outputs are written
}

// ---------------------------------------------------------------------------
// split scan with the output epilogue
//   o <- o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate)   per 128-value row
// The chain of warps 0-4 is the one above; the output rows leave through two
// warps of their own (6 and 7: TMEM lane quarters 2 and 3, rows 64..127 of
// D1), which trail the chain by up to three chunks: D1 has four buffers, and
// the issuer reuses one only after they have read it.  The four CTAs of a
// (sequence, head) hold 32 values of a row each.  Every output thread
// publishes its row's sum of squares as one tagged word (tag = chunk + 1 in
// the low half, the fp32 sum in the high half, written and read whole) in a
// ring in the workspace that the prep clears.  Warp 5 collects the four CTAs'
// words of each row (polling two chunks at a time, so that the L2 round trip
// stays off the output warps) and hands the row totals to the output warps
// through shared memory.  Output step c publishes chunk c and finishes chunk
// c - 1 with warp 5's totals.  So a thread publishes chunk c + 2 only after
// its CTA has finished chunk c, i.e. after every CTA has published chunk c,
// which each does only after finishing chunk c - 2, i.e. after its warp 5 has
// read chunk c - 2's words: in a ring of 4 slots chunk c + 2 takes chunk
// c - 2's slot once nobody reads it any more.  The grid is launched
// cooperatively, so that the four are resident together.
constexpr int kEpiScanThreads = 256;  // warps 0-4 as above; warp 5 row-sum exchange; warps 6-7 output rows
constexpr int kOutWarp0 = 6;
constexpr int kD1Bufs = 4;
constexpr uint32_t kEpiTmemCols = 256;  // D1 (4 x 32 columns), D3 (32)
static_assert(32 * kD1Bufs + BV <= (int)kEpiTmemCols, "scan TMEM columns");
static_assert(kEpiRing == 4, "the ring argument above needs four slots");
constexpr int kTotSlots = 4;                        // row totals handed from warp 5 to the output warps
constexpr int E_BAR_BYTES = 256;                    // mbarriers and the TMEM slot
static_assert(8 * (kStages + 3 + 2 * kD1Bufs + 2 * kTotSlots) + 4 <= E_BAR_BYTES, "epilogue scan barrier block");
constexpr int kGateSlots = 4;                       // gate rows prefetched two chunks ahead
constexpr int S_GATE = S_BAR + E_BAR_BYTES;         // [kGateSlots][64 rows][64 B] bf16
constexpr int S_TOT = S_GATE + kGateSlots * C * 64;  // fp32 [kTotSlots][64 rows]
constexpr int S_EPI_SMEM = S_TOT + kTotSlots * C * 4 + 1024;
static_assert(S_EPI_SMEM <= 232448, "epilogue scan shared memory");

// 16-byte copy global -> shared that completes asynchronously (commit groups)
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__global__ void __launch_bounds__(kEpiScanThreads, 1)
    chunk_scan_tc_epi_kernel(const float *__restrict__ initial_state, float *__restrict__ final_state,
                             const int32_t *__restrict__ state_indices, __nv_bfloat16 *__restrict__ o,
                             int n_seqs, int H, void *workspace, WsLayout L, EpiArgs epi) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sS = sm + S_SOP;
    unsigned char *sVn = sm + S_VOP;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + S_BAR);
    uint64_t *bar_ws = full + kStages;          // D1 = WQ S done
    uint64_t *bar_d3 = bar_ws + 1;              // D3 = KD^T Vn done
    uint64_t *bar_out = bar_d3 + 1;             // [kD1Bufs] D1 += A Vn done: the chunk's output rows
    uint64_t *bar_free = bar_out + kD1Bufs;     // [kD1Bufs] the output warps have read D1
    uint64_t *tot_full = bar_free + kD1Bufs;     // [kTotSlots] warp 5 has written a chunk's row totals
    uint64_t *tot_empty = tot_full + kTotSlots;  // [kTotSlots] the output warps have read them
    uint64_t *bar_drain = tot_empty + kTotSlots;  // exit path: every MMA issued so far is done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_drain + 1);
    float *sTot = reinterpret_cast<float *>(sm + S_TOT);
    griddep_wait();  // the records (previous kernel) are complete
    // the next forward's chunk index may be scheduled (one CTA; it waits for
    // this grid to complete before it writes anything)
    griddep_launch_dependents();

    const int n = blockIdx.x, h = blockIdx.y, vb = blockIdx.z, v0 = vb * BV;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    auto stage_of = [&](int ck) { return sm + (ck % kStages) * S_STAGE; };
    auto issue = [&](int ck) {  // the issuing thread
        unsigned char *dst = stage_of(ck);
        uint64_t *b = &full[ck % kStages];
        mbar_arrive_expect_tx(b, kStageBytes);
        bulk_g2s(dst, rec_of(ck), kImageBytes, b);
        bulk_g2s(dst + kImageBytes, rec_of(ck) + TcRec::U + vb * TcRec::UBLK, TcRec::UBLK, b);
    };

    if (warp == 0) tmem_alloc(tmem_slot, kEpiTmemCols);
    if (tid == kIssuer) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        mbar_init(bar_ws, 1);
        mbar_init(bar_d3, 1);
        for (int b = 0; b < kD1Bufs; ++b) {
            mbar_init(&bar_out[b], 1);
            mbar_init(&bar_free[b], 2);  // one arrival per output warp
        }
        for (int b = 0; b < kTotSlots; ++b) {
            mbar_init(&tot_full[b], 1);
            mbar_init(&tot_empty[b], 2);  // one arrival per output warp
        }
        mbar_init(bar_drain, 1);
        fence_mbar_init();
    }
    // state row d = tid (warps 0-3), columns v0 .. v0+31, fp32 in registers
    float S[BV];
    if (tid < D) {
#pragma unroll
        for (int x = 0; x < BV; ++x)
            S[x] = initial_state ? initial_state[st_off + (int64_t)(v0 + x) * D + tid] : 0.0f;
        store_row_n32(sS, tid, S);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tD3 = tmem + 32 * kD1Bufs;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;

    // stage loads issued / waited for by the issuer, for the exit path
    int loads_issued = 0, loads_done = 0;
    bool ok = true;
    if (warp < 5) {
        if (tid == kIssuer)
            for (int ck = 0; ck < kStages - 1 && ck < nck; ++ck, ++loads_issued) issue(ck);
        for (int ck = 0; ck < nck; ++ck) {
            const uint32_t fpar = (uint32_t)((ck / kStages) & 1), cpar = (uint32_t)(ck & 1);
            const int b = ck % kD1Bufs;
            unsigned char *st = stage_of(ck);
            const uint32_t tD1 = tmem + 32 * b;
            if (tid == kIssuer) {
                ok = mbar_wait(&full[ck % kStages], fpar) && ok;
                if (ok) loads_done = ck + 1;
                tc_fence_after();
                if (ok) {
                    mma_tile_n32<128, 128, 128>(tD1, smem_u32(st + TcRec::WQ), smem_u32(sS), false);
                    mma_commit(bar_ws);
                }
                // refill the stage of chunk ck-1 once its last MMA (D1 += A Vn) is done
                const int t = ck + kStages - 1;
                if (ok && t < nck) {
                    if (ck > 0)
                        ok = mbar_wait(&bar_out[(ck - 1) % kD1Bufs], (uint32_t)(((ck - 1) / kD1Bufs) & 1)) && ok;
                    if (ok) {
                        issue(t);
                        ++loads_issued;
                    }
                }
            } else if (warp < 2) {
                ok = mbar_wait(&full[ck % kStages], fpar) && ok;  // U of this stage
                float x[32], u[32];  // Vn = U - W S, row tid
                {  // U first, while D1 is formed
                    const uint4 *up = reinterpret_cast<const uint4 *>(st + kImageBytes + tid * 64);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        float y[8];
                        unpack8(up[c8 ^ ((tid >> 1) & 3)], y);
#pragma unroll
                        for (int t = 0; t < 8; ++t) u[8 * c8 + t] = y[t];
                    }
                }
                ok = mbar_wait(bar_ws, cpar) && ok;
                tc_fence_after();
                tmem_ld32(tD1 + lane_base, x);
                tmem_ld_wait();
#pragma unroll
                for (int vv = 0; vv < BV; ++vv) x[vv] = u[vv] - x[vv];
                store_row_n32(sVn, tid, x);
                fence_async_smem();
                tc_fence_before();
            } else if (warp < 4) {
                ok = mbar_wait(&full[ck % kStages], fpar) && ok;  // gC of this stage
            }
            // (a failure seen here is carried to the "S ready" barrier below, which
            // every state warp reaches; warps 2-3's D3 wait then gives up on its own)
            if (warp < 2 || warp == 4) ok = named_bar_and(kBarV, 96, ok);
            if (tid == kIssuer) {
                tc_fence_after();
                if (ok) {
                    mma_tile_n32<128, 64, 64, true>(tD3, smem_u32(st + TcRec::KD), smem_u32(sVn), false);
                    mma_commit(bar_d3);
                    mma_tile_n32<128, 64, 128>(tD1, smem_u32(st + TcRec::A) - 8192, smem_u32(sVn), true);
                    mma_commit(&bar_out[b]);
                }
                // the next chunk's D1 buffer last held chunk ck - 3: the output
                // warps must have read it (waited for while the state is updated)
                const int cn = ck + 1;
                if (ok && cn < nck && cn >= kD1Bufs)
                    ok = mbar_wait(&bar_free[cn % kD1Bufs], (uint32_t)(((cn / kD1Bufs) - 1) & 1)) && ok;
            } else if (warp < 4 && ok) {
                const float gc = reinterpret_cast<const float *>(st + TcRec::GC)[tid];
                ok = mbar_wait(bar_d3, cpar) && ok;
                tc_fence_after();
                float x[32];  // S = diag(gC) S + KD^T Vn
                tmem_ld32(tD3 + lane_base, x);
                tmem_ld_wait();
#pragma unroll
                for (int vv = 0; vv < BV; ++vv) S[vv] = fmaf(gc, S[vv], x[vv]);
                store_row_n32(sS, tid, S);
                fence_async_smem();
                tc_fence_before();
            }
            if (!named_bar_and(kBarS, kScanThreads, ok)) {
                ok = false;
                break;
            }
        }
    } else if (warp == 5) {

        // row totals: lane l takes rows l and l + 32 of every chunk; each round
        // reads the words of the next two chunks not yet complete
        const uint64_t *ring = ws_at<const uint64_t>(workspace, L.epi_part_off) +
                               (size_t)(n * H + h) * kEpiRing * 4 * C;  // [slot][CTA][row]
        long long tlast = clock64();  // last progress
        int cdone = 0;
        while (cdone < nck) {
            bool comp[2] = {false, false};
            float tot[2][2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = cdone + k;
                if (c >= nck) break;
                const uint64_t *slot = ring + (size_t)(c % kEpiRing) * 4 * C + lane;
                uint64_t wd[2][4];
#pragma unroll
                for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                    for (int j = 0; j < 4; ++j) wd[hr][j] = ld_relaxed_gpu_u64(slot + j * C + 32 * hr);
                bool all = true;
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    float t = 0.0f;  // summed in CTA order: the same rounding in all four
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        all = all && (uint32_t)wd[hr][j] == (uint32_t)(c + 1);
                        t += __uint_as_float((uint32_t)(wd[hr][j] >> 32));
                    }
                    tot[k][hr] = t;
                }
                comp[k] = __all_sync(0xffffffffu, all);
            }
            // hand over, in order, the chunks found complete
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (!comp[k] || (k == 1 && !comp[0])) break;
                const int c = cdone, sl = c % kTotSlots;
                if (c >= kTotSlots) ok = mbar_wait(&tot_empty[sl], (uint32_t)(((c / kTotSlots) - 1) & 1)) && ok;
                if (!ok) break;
                sTot[sl * C + lane] = tot[k][0];
                sTot[sl * C + lane + 32] = tot[k][1];
                __syncwarp();
                if (lane == 0) mbar_arrive(&tot_full[sl]);
                ++cdone;
            }
            if (!ok) break;
            // a chunk's words come about one state step apart: poll sparingly
            if (comp[0]) {
                tlast = clock64();
            } else if (clock64() - tlast > 4000000000LL) {  // no word for ~2 s
                ok = false;
                break;
            }
            __nanosleep(comp[0] ? 400 : 200);
        }
    } else if (warp >= kOutWarp0) {
        // output rows: row r of each chunk is TMEM lane 64 + r of its D1 buffer
        const int r = tid - 32 * kOutWarp0;
        const __nv_bfloat16 *gate = reinterpret_cast<const __nv_bfloat16 *>(epi.out_gate);
        uint64_t *ring = ws_at<uint64_t>(workspace, L.epi_part_off) +
                         (size_t)(n * H + h) * kEpiRing * 4 * C + r;  // [slot][CTA][row]
        float w[BV];
#pragma unroll
        for (int c4 = 0; c4 < BV / 4; ++c4) {
            const float4 wv = *reinterpret_cast<const float4 *>(epi.weight + v0 + 4 * c4);
            w[4 * c4] = wv.x;
            w[4 * c4 + 1] = wv.y;
            w[4 * c4 + 2] = wv.z;
            w[4 * c4 + 3] = wv.w;
        }
        auto row_of = [&](int ck) { return ((int64_t)start + (int64_t)ck * C + r) * H + h; };
        auto live_of = [&](int ck) { return r < min(C, len - ck * C); };
        // this thread's gate row of chunk ck: four 16-byte units in slot ck % 4,
        // unit c at c ^ ((r / 2) % 4) (conflict-free reads across the warp)
        unsigned char *grow = sm + S_GATE + r * 64;
        auto gate_unit = [&](int ck, int c8) {
            return grow + (ck % kGateSlots) * (C * 64) + ((c8 ^ ((r >> 1) & 3)) << 4);
        };
        auto fetch_gate = [&](int ck) {  // one commit group per call, empty past the end
            if (ck < nck && live_of(ck)) {
                const uint4 *gq = reinterpret_cast<const uint4 *>(gate + row_of(ck) * D + v0);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) cp_async16(gate_unit(ck, c8), gq + c8);
            }
            cp_async_commit();
        };
        fetch_gate(0);
        fetch_gate(1);
        // Step ck: chunk ck's rows into x, its sum published, chunk ck + 2's
        // gate row requested; chunk ck - 1 finished from xp with warp 5's row
        // total.  Called with the two register sets swapped on alternate
        // steps.
        auto step = [&](int ck, float (&x)[BV], float (&xp)[BV]) -> bool {
            fetch_gate(ck + 2);
            if (ck > 0) {
                cp_async_wait<3>();  // chunk ck - 1's gate row (groups ck, ck + 1, ck + 2 may be pending)
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float gv[8];
                    unpack8(live_of(ck - 1) ? *reinterpret_cast<const uint4 *>(gate_unit(ck - 1, c8))
                                            : make_uint4(0, 0, 0, 0),
                            gv);
#pragma unroll
                    for (int t = 0; t < 8; ++t)  // sigmoid(g) = 1 / (1 + e^-g)
                        xp[8 * c8 + t] *= w[8 * c8 + t] * __fdividef(1.0f, 1.0f + __expf(-gv[t]));
                }
            }
            if (ck < nck) {
                const int b = ck % kD1Bufs;
                if (!mbar_wait(&bar_out[b], (uint32_t)((ck / kD1Bufs) & 1))) return false;
                tc_fence_after();
                tmem_ld32(tmem + 32 * b + lane_base, x);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_free[b]);  // D1[b] may be reused
                float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // rows past the sequence end are zero
#pragma unroll
                for (int vv = 0; vv < BV; ++vv) s4[vv & 3] = fmaf(x[vv], x[vv], s4[vv & 3]);
                const float ss = (s4[0] + s4[1]) + (s4[2] + s4[3]);
                st_relaxed_gpu_u64(ring + (size_t)(ck % kEpiRing) * 4 * C + vb * C,
                                   ((uint64_t)__float_as_uint(ss) << 32) | (uint32_t)(ck + 1));
            }
            if (ck > 0) {
                const int sl = (ck - 1) % kTotSlots;
                if (!mbar_wait(&tot_full[sl], (uint32_t)(((ck - 1) / kTotSlots) & 1))) return false;
                const float tot = sTot[sl * C + r];
                __syncwarp();
                if (lane == 0) mbar_arrive(&tot_empty[sl]);
                const float rn = rsqrtf(tot * (1.0f / D) + epi.eps);
                if (live_of(ck - 1)) {
                    uint4 *op = reinterpret_cast<uint4 *>(o + row_of(ck - 1) * D + v0);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        float y[8];
#pragma unroll
                        for (int t = 0; t < 8; ++t) y[t] = xp[8 * c8 + t] * rn;
                        op[c8] = pack8(y);
                    }
                }
            }
            return true;
        };
        float xa[BV], xb[BV];
        for (int ck = 0; ck <= nck && ok; ck += 2) {
            ok = step(ck, xa, xb);
            if (ok && ck + 1 <= nck) ok = step(ck + 1, xb, xa);
        }
        cp_async_wait<0>();  // nothing in flight into shared memory at exit
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        // let copies and MMAs still in flight land before the shared memory
        // and the TMEM are released
        if (tid == kIssuer) {
            atomicOr(status, kStatusTimeout);
            for (int t = loads_done; t < loads_issued; ++t)
                mbar_wait(&full[t % kStages], (uint32_t)((t / kStages) & 1), 400000000LL);
            mma_commit(bar_drain);
            mbar_wait(bar_drain, 0, 400000000LL);
        }
    } else if (final_state && tid < D) {
#pragma unroll
        for (int x = 0; x < BV; ++x) final_state[st_off + (int64_t)(v0 + x) * D + tid] = S[x];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kEpiTmemCols);
}

// ---------------------------------------------------------------------------
// wide scan: one CTA per (sequence, head) covering all 128 value columns.
// An MMA instruction costs the same for N = 32 and N = 128, so this does a
// split scan's per-chunk MMA work for four times the columns; it is the
// better choice once sequences x heads x 4 exceed the SM count.
// ---------------------------------------------------------------------------
constexpr int kWideThreads = 288;  // warps 0-7: (TMEM quarter, column half); warp 8: MMAs and loads
constexpr int kWideIssuer = 256;
constexpr int kWideStages = 2;
constexpr uint32_t kWideTmemCols = 512;  // D1 double-buffered (2 x 128 columns), D3 (128)
constexpr uint32_t kWideStageBytes = TcRec::U + 4 * TcRec::UBLK;  // the whole record
constexpr int W_STAGE = 74752;                                    // rounded up to 1024
constexpr int W_SOP = kWideStages * W_STAGE;  // S operand [128 keys][128] bf16, MN-major SW128, 32 KB
constexpr int W_VOP = W_SOP + 32768;          // Vn operand [64 rows][128] bf16, MN-major SW128, 16 KB
constexpr int W_BAR = W_VOP + 16384;          // full[kWideStages], ws, d3, out, drain, tmem slot
constexpr int W_SMEM = W_BAR + 64 + 1024;
static_assert(kWideStageBytes <= (uint32_t)W_STAGE && W_STAGE % 1024 == 0, "wide stage");
static_assert(kWideStageBytes % 16 == 0, "bulk copy size");
static_assert(W_SMEM <= 232448, "wide scan shared memory");

__global__ void __launch_bounds__(kWideThreads, 1)
    chunk_scan_wide_kernel(const float *__restrict__ initial_state, float *__restrict__ final_state,
                           const int32_t *__restrict__ state_indices, __nv_bfloat16 *__restrict__ o,
                           int n_seqs, int H, void *workspace, WsLayout L) {
    griddep_wait();  // the records (previous kernel) are complete
    // the next forward's chunk index may be scheduled (one CTA; it waits for
    // this grid to complete before it writes anything)
    griddep_launch_dependents();
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sS = sm + W_SOP;
    unsigned char *sVn = sm + W_VOP;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + W_BAR);
    uint64_t *bar_ws = full + kWideStages;  // D1 = WQ S done
    uint64_t *bar_d3 = bar_ws + 1;          // D3 = KD^T Vn done
    uint64_t *bar_out = bar_d3 + 1;         // D1 += A Vn done: the chunk's output rows
    uint64_t *bar_drain = bar_out + 1;      // exit path: every MMA issued so far is done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_drain + 1);

    // longest sequences first: the grid walks the sequences by decreasing
    // length, all heads of one sequence before the next
    const int n = ws_at<const int32_t>(workspace, L.seq_order_off)[blockIdx.x / H], h = blockIdx.x % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, half = (warp >> 2) & 1;  // TMEM lane quarter, value-column half
    const int32_t start = ws_at<const int32_t>(workspace, L.seq_start_off)[n];
    if (start < 0) return;  // sequence skipped (bad cu_seqlens or slot)
    const int len = ws_at<const int32_t>(workspace, L.seq_len_off)[n];
    const int c0 = ws_at<const int32_t>(workspace, L.chunk_off_off)[n];
    const int nck = (len + C - 1) / C;
    const int64_t slot = state_indices ? (int64_t)state_indices[n] : (int64_t)n;
    const int64_t st_off = (slot * H + h) * (int64_t)D * D;  // [V][K] block of (slot, h)
    int32_t *status = ws_at<int32_t>(workspace, L.status_off);
    const unsigned char *recs = ws_at<const unsigned char>(workspace, L.records_off);
    auto stage_of = [&](int ck) { return sm + (ck % kWideStages) * W_STAGE; };
    auto issue = [&](int ck) {  // the issuing thread
        uint64_t *b = &full[ck % kWideStages];
        mbar_arrive_expect_tx(b, kWideStageBytes);
        bulk_g2s(stage_of(ck), recs + ((size_t)(c0 + ck) * H + h) * TcRec::bytes, kWideStageBytes, b);
    };

    if (warp == 0) tmem_alloc(tmem_slot, kWideTmemCols);
    if (tid == kWideIssuer) {
        for (int s = 0; s < kWideStages; ++s) mbar_init(&full[s], 1);
        mbar_init(bar_ws, 1);
        mbar_init(bar_d3, 1);
        mbar_init(bar_out, 1);
        mbar_init(bar_drain, 1);
        fence_mbar_init();
    }
    // state row d = 32 q + lane, value columns 64 half .. 64 half + 63, fp32
    const int d = 32 * q + lane, vh = 64 * half;
    float S[64];
    auto store_s = [&]() {  // this thread's part of the S operand (MN-major [d][v])
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float y[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) y[t] = S[8 * c + t];
            *reinterpret_cast<uint4 *>(sS + sw128_off(d, vh + 8 * c, D)) = pack8(y);
        }
    };
    if (warp < 8) {
#pragma unroll
        for (int x = 0; x < 64; ++x)
            S[x] = initial_state ? initial_state[st_off + (int64_t)(vh + x) * D + d] : 0.0f;
        store_s();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tD3 = tmem + 256;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;

    // output rows 64 + 32 (q - 2) + lane of chunk ck (TMEM D1 buffer ck & 1), this half
    auto store_output = [&](int ck) {
        const int r = 32 * (q - 2) + lane;
        const bool live = r < min(C, len - ck * C);
        const int64_t tok = (int64_t)start + (int64_t)ck * C + r;
        uint4 *op = reinterpret_cast<uint4 *>(o + (tok * H + h) * (int64_t)D + vh);
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            float x[32];
            tmem_ld32(tmem + 128 * (ck & 1) + vh + 32 * p + lane_base, x);
            tmem_ld_wait();
            if (live) {
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t];
                    op[4 * p + c8] = pack8(y);
                }
            }
        }
    };

    int loads_issued = 0, loads_done = 0;
    if (tid == kWideIssuer && nck > 0) {
        issue(0);
        loads_issued = 1;
    }
    bool ok = true;
    for (int ck = 0; ck < nck; ++ck) {
        const uint32_t fpar = (uint32_t)((ck / kWideStages) & 1), cpar = (uint32_t)(ck & 1);
        unsigned char *st = stage_of(ck);
        const uint32_t tD1 = tmem + 128 * (ck & 1);
        if (tid == kWideIssuer) {
            ok = mbar_wait(&full[ck % kWideStages], fpar) && ok;
            if (ok) loads_done = ck + 1;
            tc_fence_after();
            if (ok) {
                mma_tile<128, 128, 128, 128, 128, false, true>(tD1, smem_u32(st + TcRec::WQ), smem_u32(sS), false);
                mma_commit(bar_ws);
            }
            // next chunk into the other stage once chunk ck-1's last MMA is done
            if (ok && ck + 1 < nck) {
                if (ck > 0) ok = mbar_wait(bar_out, cpar ^ 1) && ok;
                if (ok) {
                    issue(ck + 1);
                    ++loads_issued;
                }
            }
        } else if (warp < 8) {
            ok = mbar_wait(&full[ck % kWideStages], fpar) && ok;  // U and gC of this stage
            if (q < 2) {  // Vn = U - W S, row j = d, this half of the columns
                ok = mbar_wait(bar_ws, cpar) && ok;
                tc_fence_after();
                const int j = d;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    float x[32], u[32];
                    tmem_ld32(tD1 + vh + 32 * p + lane_base, x);
                    const uint4 *up = reinterpret_cast<const uint4 *>(st + TcRec::U + (2 * half + p) * TcRec::UBLK + j * 64);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        float y[8];
                        unpack8(up[c8 ^ ((j >> 1) & 3)], y);
#pragma unroll
                        for (int t = 0; t < 8; ++t) u[8 * c8 + t] = y[t];
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        float y[8];
#pragma unroll
                        for (int t = 0; t < 8; ++t) y[t] = u[8 * c8 + t] - x[8 * c8 + t];
                        *reinterpret_cast<uint4 *>(sVn + sw128_off(j, vh + 32 * p + 8 * c8, C)) = pack8(y);
                    }
                }
                fence_async_smem();
            } else if (ck > 0) {  // output rows of the previous chunk
                ok = mbar_wait(bar_out, cpar ^ 1) && ok;
                tc_fence_after();
                if (ok) store_output(ck - 1);
            }
            tc_fence_before();
        }
        // (a failure seen here is carried to the "S ready" barrier below, which
        // every warp reaches.)  The output warps meet "Vn ready" too: they wait
        // on bar_out's phase of chunk ck-1 by parity, so the issuer must not
        // complete chunk ck's phase (D1 += A Vn, issued after this barrier)
        // before they have seen the previous one.
        ok = named_bar_and(kBarV, kWideThreads, ok);
        if (tid == kWideIssuer) {
            tc_fence_after();
            if (ok) {
                mma_tile<128, 128, 64, 64, 64, true, true>(tD3, smem_u32(st + TcRec::KD), smem_u32(sVn), false);
                mma_commit(bar_d3);
                mma_tile<128, 128, 64, 128, 64, false, true>(tD1, smem_u32(st + TcRec::A) - 8192, smem_u32(sVn), true);
                mma_commit(bar_out);
            }
        } else if (warp < 8 && ok) {
            const float gc = reinterpret_cast<const float *>(st + TcRec::GC)[d];
            ok = mbar_wait(bar_d3, cpar) && ok;
            tc_fence_after();
#pragma unroll
            for (int p = 0; p < 2; ++p) {  // S = diag(gC) S + KD^T Vn
                float x[32];
                tmem_ld32(tD3 + vh + 32 * p + lane_base, x);
                tmem_ld_wait();
#pragma unroll
                for (int vv = 0; vv < 32; ++vv) S[32 * p + vv] = fmaf(gc, S[32 * p + vv], x[vv]);
            }
            store_s();
            fence_async_smem();
            tc_fence_before();
        }
        if (!named_bar_and(kBarS, kWideThreads, ok)) {
            ok = false;
            break;
        }
    }
    if (ok && nck > 0 && warp < 8 && q >= 2) {
        ok = mbar_wait(bar_out, (uint32_t)((nck - 1) & 1));
        tc_fence_after();
        if (ok) store_output(nck - 1);
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (tid == kWideIssuer) {
            atomicOr(status, kStatusTimeout);
            for (int t = loads_done; t < loads_issued; ++t)
                mbar_wait(&full[t % kWideStages], (uint32_t)((t / kWideStages) & 1), 400000000LL);
            mma_commit(bar_drain);
            mbar_wait(bar_drain, 0, 400000000LL);
        }
    } else if (final_state && warp < 8) {
#pragma unroll
        for (int x = 0; x < 64; ++x) final_state[st_off + (int64_t)(vh + x) * D + d] = S[x];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kWideTmemCols);
}

}  // namespace

cudaError_t launch_chunk_prep_tc(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const GateArgs *gate, int n_seqs,
                                 int64_t total_tokens, int H, float scale, int scan_ctas,
                                 void *workspace, cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, TcRec::bytes);
    const int64_t items_max = max_chunks(total_tokens, n_seqs) * (int64_t)H;
    // two CTAs per SM; beside a scan that runs alongside, one on each of its SMs
    const int grid = (int)std::min<int64_t>(items_max, (int64_t)kPrepMinBlocks * sm_count() - scan_ctas);
    RawMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (total_tokens > 0) {
        if (!encode_rows(&maps.q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens, true) ||
            !encode_rows(&maps.k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens, true) ||
            !encode_rows(&maps.v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens, true) ||
            !(gate ? encode_rows(&maps.g, gate->raw_gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens)
                   : encode_rows(&maps.g, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, total_tokens)))
            return cudaErrorInvalidValue;
    }
    GateArgs ga;
    memset(&ga, 0, sizeof(ga));
    if (gate) ga = *gate;
    auto kern = gate ? chunk_prep_tc_kernel<true> : chunk_prep_tc_kernel<false>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    cudaError_t e = launch_dependent(kern, dim3(grid), dim3(kPrepThreads), P_SMEM, stream, maps, g,
                                     beta, ga, n_seqs, H, scale, scan_ctas, workspace, L);
    if (e == cudaSuccess) e = cudaGetLastError();
    // the items deferred above (none in most workloads: its CTAs then exit at once)
    if (e == cudaSuccess)
        e = launch_chunk_prep_tc_strong(q, k, v, g, beta, gate, n_seqs, total_tokens, H, scale,
                                        scan_ctas, grid, workspace, stream);
    return e;
}

cudaError_t launch_chunk_scan_tc(const float *initial_state, float *final_state,
                                 const int32_t *state_indices, void *o, int n_seqs,
                                 int64_t total_tokens, int H, int flags, const EpiArgs *epi,
                                 bool *epi_applied, void *workspace, cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, TcRec::bytes);
    *epi_applied = false;
    // wide scan once four CTAs per (sequence, head) would not fit in one wave
    const bool wide = (flags & KDA_CHUNK_SCAN_WIDE) ||
                      (!(flags & KDA_CHUNK_SCAN_SPLIT) && (int64_t)n_seqs * H * (D / BV) > sm_count());
    if (wide) {
        const dim3 grid((unsigned)((int64_t)n_seqs * H), 1, 1);
        cudaFuncSetAttribute(chunk_scan_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, W_SMEM);
        const cudaError_t e = launch_dependent(chunk_scan_wide_kernel, grid, dim3(kWideThreads), W_SMEM,
                                               stream, initial_state, final_state, state_indices,
                                               (__nv_bfloat16 *)o, n_seqs, H, workspace, L);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const dim3 grid((unsigned)n_seqs, (unsigned)H, D / BV);
    const int64_t ctas = (int64_t)n_seqs * H * (D / BV);
    // the epilogue in the scan: 16-byte aligned gate rows, exchange room for
    // every (sequence, head), and the whole grid resident at once
    bool fuse = epi && epi->out_gate && ((uintptr_t)epi->out_gate % 16 == 0) &&
                (int64_t)n_seqs * H <= kEpiPairs;
    if (fuse) {
        int per_sm = 0;
        cudaFuncSetAttribute(chunk_scan_tc_epi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S_EPI_SMEM);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chunk_scan_tc_epi_kernel, kEpiScanThreads,
                                                          S_EPI_SMEM) != cudaSuccess) {
            cudaGetLastError();
            per_sm = 0;
        }
        fuse = ctas <= (int64_t)per_sm * sm_count();
    }
    if (fuse) {
        const cudaError_t e = launch_dependent_coop(chunk_scan_tc_epi_kernel, grid, dim3(kEpiScanThreads),
                                                    S_EPI_SMEM, stream, initial_state, final_state, state_indices,
                                                    (__nv_bfloat16 *)o, n_seqs, H, workspace, L, *epi);
        if (e == cudaSuccess) {
            *epi_applied = true;
            return cudaGetLastError();
        }
        // a cooperative launch refused here (nothing was launched): the plain
        // split scan below, and the separate pass after it
        cudaGetLastError();
    }
    cudaFuncSetAttribute(chunk_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S_SMEM);
    const cudaError_t e = launch_dependent(chunk_scan_tc_kernel, grid, dim3(kSplitThreads), S_SMEM, stream,
                                           initial_state, final_state, state_indices, (__nv_bfloat16 *)o,
                                           n_seqs, H, workspace, L);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

void preload_chunk_tc_kernels() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, chunk_prep_tc_kernel<true>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, chunk_prep_tc_kernel<false>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, chunk_scan_tc_overlap_kernel) != cudaSuccess)
        cudaGetLastError();
}

int launch_chunk_scan_tc_ahead(const float *initial_state, float *final_state,
                               const int32_t *state_indices, void *o, int n_seqs,
                               int64_t total_tokens, int H, int flags, const EpiArgs *epi,
                               void *workspace, cudaStream_t stream, cudaError_t *err) {
    (void)epi;  // with an epilogue, the separate pass follows the step
    *err = cudaSuccess;
    const int64_t ctas = (int64_t)n_seqs * H * (D / BV);
    // the split layout, one CTA per SM, and SMs left over for the strong-decay
    // prep (which cannot share an SM with a scan CTA) and for prep CTAs in pairs
    if ((flags & KDA_CHUNK_SCAN_WIDE) || ctas + 8 > sm_count()) return 0;
    {  // every kernel launched while this scan runs is loaded first (once per device)
        static bool loaded[64] = {false};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
            cudaGetLastError();
            return 0;
        }
        if (!loaded[dev]) {
            preload_chunk_tc_kernels();
            preload_chunk_tc_strong_kernels();
            preload_chunk_index_kernel();
            preload_output_gate_norm_kernels();
            loaded[dev] = true;
        }
    }
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, TcRec::bytes);
    const dim3 grid((unsigned)n_seqs, (unsigned)H, D / BV);
    cudaFuncSetAttribute(chunk_scan_tc_overlap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SP_SMEM);
    // the whole 228 KB as shared memory, so that a prep CTA fits beside a scan CTA
    cudaFuncSetAttribute(chunk_scan_tc_overlap_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    // cooperative: every CTA is resident before the prep (launched next, and
    // let go once every scan CTA has started) takes the rest of the GPU
    const cudaError_t e = launch_dependent_coop(chunk_scan_tc_overlap_kernel, grid, dim3(kSplitThreads), SP_SMEM,
                                                stream, initial_state, final_state, state_indices,
                                                (__nv_bfloat16 *)o, n_seqs, H, workspace, L);
    if (e != cudaSuccess) {  // refused (nothing was launched): the scan runs after the prep
        cudaGetLastError();
        return 0;
    }
    *err = cudaGetLastError();
    return (int)ctas;
}

}  // namespace kda
