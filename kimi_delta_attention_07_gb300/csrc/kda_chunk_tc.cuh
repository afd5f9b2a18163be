// Helpers shared by the tensor-core chunk kernels (kda_chunk_tc.cu and
// kda_chunk_tc_strong.cu): bf16 packing, the model's gate with SFU
// intrinsics, and the host-side encoder of the TMA tensor maps over the
// [T, H, 128] activations.
#pragma once

#include <cuda.h>  // CUtensorMap (the encoder is fetched through the runtime)
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
}

__device__ __forceinline__ float2 unpack2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}

// 8 consecutive bf16 (16 bytes) -> fp32
__device__ __forceinline__ void unpack8(uint4 raw, float (&x)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2(w[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// The model's gate (see gate_decay) with the SFU exponential, logarithm and
// reciprocal (a few ulp, far below the bf16 operands of this path); log1p of
// a small argument by its series, where 1 + e would round the argument away.
__device__ __forceinline__ float gate_decay_fast(float x, float gscale, float lower_bound,
                                                 bool use_lower_bound) {
    if (use_lower_bound) return __fdividef(lower_bound, 1.0f + __expf(-gscale * x));
    const float e = __expf(-fabsf(x));  // in (0, 1]
    const float l1p = e < 1e-3f ? e * (1.0f - 0.5f * e) : __logf(1.0f + e);
    return -gscale * (fmaxf(x, 0.0f) + l1p);
}

// ---- host: TMA tensor maps -------------------------------------------------------

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 3-D map {128, H, T} over a [T, H, 128] tensor with 64-token boxes: either
// 128 channels per box, no swizzle (swizzled64 = false), or 64 channels per
// box (128 bytes of bf16) with 128-byte swizzle, i.e. a K-major or MN-major
// SW128 operand tile of 64 rows.
inline bool encode_rows(CUtensorMap *m, const void *base, CUtensorMapDataType dt, size_t elem,
                        int H, int64_t T, bool swizzled64 = false) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)(kHeadDim * elem),
                                   (cuuint64_t)(kHeadDim * elem) * (cuuint64_t)H};
    const cuuint32_t box[3] = {(cuuint32_t)(swizzled64 ? 64 : kHeadDim), 1, (cuuint32_t)kChunk};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzled64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace kda
