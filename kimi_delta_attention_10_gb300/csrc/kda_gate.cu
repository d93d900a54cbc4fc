// kda_gate: g = -exp(A_log[h]) * softplus(f + dt_bias[h, c]) and beta = sigmoid(b).
//
// The decay is formed outside the chunk kernel with FP32 A_log/dt_bias, and
// beta is the sigmoid of its logits ("GLM-5.3-Flash F6.2: KDA correctness and
// FLA sequence parallelism", fused-gate commit).
//
// HBM-bound elementwise kernel: each thread moves 4 consecutive channels
// (one 16-byte FP32 store, a 16- or 8-byte load), grid-stride over the
// [T, H, K] tensor; the [T, H] beta tensor is a second grid-stride loop in
// the same launch.  Algorithmic bytes: T*H*K*(sizeof f + 4) + T*H*(sizeof b + 4).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

__device__ __forceinline__ float4 load4(const float* p, int64_t i)
{
    return __ldcs(reinterpret_cast<const float4*>(p + i));
}

__device__ __forceinline__ float4 load4(const __nv_bfloat16* p, int64_t i)
{
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p + i));
    float4 r;
    r.x = __uint_as_float(u.x << 16);
    r.y = __uint_as_float(u.x & 0xffff0000u);
    r.z = __uint_as_float(u.y << 16);
    r.w = __uint_as_float(u.y & 0xffff0000u);
    return r;
}

template <typename TF, typename TB>
__global__ void __launch_bounds__(256) gate_kernel(const TF* __restrict__ f,
                                                   const float* __restrict__ A_log,
                                                   const float* __restrict__ dt_bias,
                                                   const TB* __restrict__ b, int64_t T,
                                                   int32_t H, int32_t K,
                                                   float* __restrict__ g_out,
                                                   float* __restrict__ beta_out)
{
    const int64_t n4 = T * H * (int64_t)K / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int32_t K4 = K / 4;
    for (int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i4 < n4; i4 += stride) {
        const int64_t row = i4 / K4;                    // t * H + h
        const int32_t c = (int32_t)(i4 - row * K4) * 4;
        const int32_t h = (int32_t)(row % H);
        const float lam = -expf(__ldg(A_log + h));
        const float4 x = load4(f, i4 * 4);
        const float4 db = __ldg(reinterpret_cast<const float4*>(dt_bias + (int64_t)h * K + c));
        float4 r;
        r.x = gate_decay(x.x, db.x, lam);
        r.y = gate_decay(x.y, db.y, lam);
        r.z = gate_decay(x.z, db.z, lam);
        r.w = gate_decay(x.w, db.w, lam);
        __stcs(reinterpret_cast<float4*>(g_out + i4 * 4), r);
    }
    const int64_t nb = T * H;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nb; i += stride) {
        const float x = load_as_float(b + i);
        beta_out[i] = gate_sigmoid(x);
    }
}

template <typename TF, typename TB>
cudaError_t launch_typed(const void* f, const float* A_log, const float* dt_bias, const void* b,
                         int64_t T, int32_t H, int32_t K, float* g_out, float* beta_out,
                         cudaStream_t stream)
{
    const int64_t n4 = T * H * (int64_t)K / 4;
    const int sms = device_sm_count();
    const int64_t max_blocks = (int64_t)(sms > 0 ? sms : 152) * 8;   // 8 x 256 threads per SM
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > max_blocks) blocks = max_blocks;
    if (blocks < 1) blocks = 1;
    gate_kernel<TF, TB><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const TF*>(f), A_log, dt_bias, static_cast<const TB*>(b), T, H, K, g_out,
        beta_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate(const void* f, bool f_bf16, const float* A_log, const float* dt_bias,
                        const void* b, bool b_bf16, int64_t T, int32_t H, int32_t K,
                        float* g_out, float* beta_out, cudaStream_t stream)
{
    if (f_bf16) {
        return b_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(f, A_log, dt_bias, b, T, H, K,
                                                                   g_out, beta_out, stream)
                      : launch_typed<__nv_bfloat16, float>(f, A_log, dt_bias, b, T, H, K, g_out,
                                                           beta_out, stream);
    }
    return b_bf16 ? launch_typed<float, __nv_bfloat16>(f, A_log, dt_bias, b, T, H, K, g_out,
                                                       beta_out, stream)
                  : launch_typed<float, float>(f, A_log, dt_bias, b, T, H, K, g_out, beta_out,
                                               stream);
}

}  // namespace kda
