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
__global__ void __launch_bounds__(kEpiThreads)
    output_gate_norm_kernel(T *__restrict__ o, const EpiArgs epi, int64_t rows) {
    const int lane = threadIdx.x & 31;
    const float4 w = *reinterpret_cast<const float4 *>(epi.weight + 4 * lane);
    const T *gate = reinterpret_cast<const T *>(epi.out_gate);
    const int64_t warps = (int64_t)gridDim.x * (kEpiThreads / 32);
    for (int64_t r = blockIdx.x * (int64_t)(kEpiThreads / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
        const int64_t e = r * kHeadDim + 4 * lane;
        const float4 x = load4(o + e);
        const float4 gt = load4(gate + e);
        const float ms = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w) * (1.0f / kHeadDim);
        const float rn = 1.0f / sqrtf(ms + epi.eps);
        store4(o + e, make_float4(x.x * rn * w.x * gate_beta(gt.x), x.y * rn * w.y * gate_beta(gt.y),
                                  x.z * rn * w.z * gate_beta(gt.z), x.w * rn * w.w * gate_beta(gt.w)));
    }
}

}  // namespace

cudaError_t launch_output_gate_norm(void *o, const EpiArgs &epi, int64_t rows, int dtype,
                                    cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + (kEpiThreads / 32) - 1) / (kEpiThreads / 32);
    const int grid = (int)std::min<int64_t>(blocks, 152 * 16);
    if (dtype == KDA_BF16)
        output_gate_norm_kernel<__nv_bfloat16><<<grid, kEpiThreads, 0, stream>>>(
            (__nv_bfloat16 *)o, epi, rows);
    else
        output_gate_norm_kernel<float><<<grid, kEpiThreads, 0, stream>>>((float *)o, epi, rows);
    return cudaGetLastError();
}

}  // namespace kda
