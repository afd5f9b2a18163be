// The model's output epilogue (Ascend model file, KimiDeltaAttention.
// _project_out): per (token, head) row of V = 128 values,
//   o <- o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate)
// in place, one warp per row (4 values per lane, a shuffle reduction).  HBM
// bound: o read and written once, the gate read once.
#include <algorithm>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kEpiThreads = 256;

template <typename T>
__device__ __forceinline__ void store4(T *p, float4 x);
template <>
__device__ __forceinline__ void store4<float>(float *p, float4 x) {
    *reinterpret_cast<float4 *>(p) = x;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, float4 x) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

template <typename T>
__device__ __forceinline__ float4 gated_row(float4 x, float4 gt, float4 w, float eps) {
    const float ms = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w) * (1.0f / kHeadDim);
    const float rn = 1.0f / sqrtf(ms + eps);
    return make_float4(x.x * rn * w.x * gate_beta(gt.x), x.y * rn * w.y * gate_beta(gt.y),
                       x.z * rn * w.z * gate_beta(gt.z), x.w * rn * w.w * gate_beta(gt.w));
}

// One warp per row; a warp takes two rows (r and r + warps) per step and
// issues all four loads before the first store, so that two rows of each
// warp are in flight.  The grid is the resident one (a grid-stride loop).
template <typename T>
__global__ void __launch_bounds__(kEpiThreads)
    output_gate_norm_kernel(T *__restrict__ o, const EpiArgs epi, int64_t rows) {
    // launched as a dependent of the kernel before it (the scan, or the
    // strong-decay prep that finishes after the scan): scheduled early, it
    // reads o once that kernel has completed
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const float4 w = *reinterpret_cast<const float4 *>(epi.weight + 4 * lane);
    const T *__restrict__ gate = reinterpret_cast<const T *>(epi.out_gate);
    const int64_t warps = (int64_t)gridDim.x * (kEpiThreads / 32);
    int64_t r = blockIdx.x * (int64_t)(kEpiThreads / 32) + (threadIdx.x >> 5);
    for (; r + warps < rows; r += 2 * warps) {
        const int64_t e0 = r * kHeadDim + 4 * lane, e1 = e0 + warps * kHeadDim;
        const float4 x0 = load4(o + e0), g0 = load4(gate + e0);
        const float4 x1 = load4(o + e1), g1 = load4(gate + e1);
        store4(o + e0, gated_row<T>(x0, g0, w, epi.eps));
        store4(o + e1, gated_row<T>(x1, g1, w, epi.eps));
    }
    if (r < rows) {
        const int64_t e = r * kHeadDim + 4 * lane;
        store4(o + e, gated_row<T>(load4(o + e), load4(gate + e), w, epi.eps));
    }
}

}  // namespace

void preload_output_gate_norm_kernels() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, output_gate_norm_kernel<__nv_bfloat16>) != cudaSuccess ||
        cudaFuncGetAttributes(&a, output_gate_norm_kernel<float>) != cudaSuccess)
        cudaGetLastError();
}

cudaError_t launch_output_gate_norm(void *o, const EpiArgs &epi, int64_t rows, int dtype,
                                    cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + (kEpiThreads / 32) - 1) / (kEpiThreads / 32);
    // one wave of resident blocks, so that no block waits for a second wave
    auto one_wave = [&](auto kernel) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kEpiThreads, 0) !=
                cudaSuccess ||
            per_sm < 1) {
            cudaGetLastError();
            per_sm = 1;
        }
        return (int)std::min<int64_t>(blocks, (int64_t)sm_count() * per_sm);
    };
    cudaError_t e;
    if (dtype == KDA_BF16) {
        auto kern = output_gate_norm_kernel<__nv_bfloat16>;
        e = launch_dependent(kern, dim3(one_wave(kern)), dim3(kEpiThreads), 0, stream,
                             (__nv_bfloat16 *)o, epi, rows);
    } else {
        auto kern = output_gate_norm_kernel<float>;
        e = launch_dependent(kern, dim3(one_wave(kern)), dim3(kEpiThreads), 0, stream, (float *)o, epi,
                             rows);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kda
