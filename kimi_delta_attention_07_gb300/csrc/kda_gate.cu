// The model's gate activation into fp32 buffers, for gated calls on the fp32
// chunk path (the tensor-core path activates the raw gate on chip instead).
// Ascend model file, _prefill_torch_kda: x = raw_gate + dt_bias[h][k];
// g = lower_bound * sigmoid(exp(A_log[h]) x) or -exp(A_log[h]) softplus(x);
// beta = sigmoid(raw_beta).
#include <algorithm>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kGateThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kGateThreads)
    gate_activation_kernel(const GateArgs gate, int64_t total_tokens, int H,
                           float *__restrict__ g_out, float *__restrict__ beta_out) {
    const T *raw = reinterpret_cast<const T *>(gate.raw_gate);
    const T *rawb = reinterpret_cast<const T *>(gate.raw_beta);
    const bool lb = gate.use_lower_bound != 0;
    const int64_t n4 = total_tokens * H * (kHeadDim / 4);  // groups of 4 channels
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = 4 * i;
        const int hk = (int)(e % ((int64_t)H * kHeadDim));  // h * K + k
        const float gs = expf(gate.a_log[hk / kHeadDim]);
        const float4 r = load4(raw + e);
        const float4 c = *reinterpret_cast<const float4 *>(gate.dt_bias + hk);
        *reinterpret_cast<float4 *>(g_out + e) =
            make_float4(gate_decay(r.x + c.x, gs, gate.lower_bound, lb),
                        gate_decay(r.y + c.y, gs, gate.lower_bound, lb),
                        gate_decay(r.z + c.z, gs, gate.lower_bound, lb),
                        gate_decay(r.w + c.w, gs, gate.lower_bound, lb));
    }
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total_tokens * H;
         i += (int64_t)gridDim.x * blockDim.x)
        beta_out[i] = gate_beta(to_f32(rawb[i]));
}

}  // namespace

cudaError_t launch_gate_activation(const GateArgs &gate, int dtype, int64_t total_tokens, int H,
                                   float *g_out, float *beta_out, cudaStream_t stream) {
    if (total_tokens == 0) return cudaSuccess;
    const int64_t n4 = total_tokens * H * (kHeadDim / 4);
    const int grid = (int)std::min<int64_t>((n4 + kGateThreads - 1) / kGateThreads, 152 * 16);
    if (dtype == KDA_BF16)
        gate_activation_kernel<__nv_bfloat16><<<grid, kGateThreads, 0, stream>>>(
            gate, total_tokens, H, g_out, beta_out);
    else
        gate_activation_kernel<float><<<grid, kGateThreads, 0, stream>>>(gate, total_tokens, H,
                                                                          g_out, beta_out);
    return cudaGetLastError();
}

}  // namespace kda
