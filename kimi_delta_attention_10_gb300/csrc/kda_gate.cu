// kda_gate: g = -exp(A_log[h]) * softplus(f + dt_bias[h, c]) and beta = sigmoid(b).
//
// The decay is formed outside the chunk kernel with FP32 A_log/dt_bias, and
// beta is the sigmoid of its logits ("GLM-5.3-Flash F6.2: KDA correctness and
// FLA sequence parallelism", fused-gate commit).
//
// HBM-bound elementwise kernel: each thread moves 4 consecutive channels
// (one 16-byte FP32 store, a 16- or 8-byte load) per element group,
// grid-stride over the [T, H, K] tensor with two groups in flight; the [T, H]
// beta tensor is a second grid-stride loop in the same launch.  Algorithmic bytes: T*H*K*(sizeof f + 4) + T*H*(sizeof b + 4).
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
    // The (head, channel group) of element i4 = (t H + h) K4 + c4 advances by a
    // fixed step per grid stride: no division inside the loop.
    const int64_t start = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int32_t c4 = (int32_t)(start % K4);
    int32_t h = (int32_t)((start / K4) % H);
    const int32_t dc4 = (int32_t)(stride % K4);
    const int32_t dh = (int32_t)((stride / K4) % H);
    auto advance = [&](int32_t& cc, int32_t& hh) {
        cc += dc4;
        const int32_t carry = cc >= K4;
        cc -= carry ? K4 : 0;
        hh += dh + carry;
        hh -= hh >= H ? H : 0;
    };
    auto decay4 = [&](int64_t i4, int32_t cc, int32_t hh) {
        const float lam = -expf(__ldg(A_log + hh));
        const float4 x = load4(f, i4 * 4);
        const float4 db = __ldg(reinterpret_cast<const float4*>(dt_bias + (int64_t)hh * K + 4 * cc));
        float4 r;
        r.x = gate_decay(x.x, db.x, lam);
        r.y = gate_decay(x.y, db.y, lam);
        r.z = gate_decay(x.z, db.z, lam);
        r.w = gate_decay(x.w, db.w, lam);
        __stcs(reinterpret_cast<float4*>(g_out + i4 * 4), r);
    };
    int64_t i4 = start;
    // two grid strides per iteration: two loads in flight per thread
    for (; i4 + stride < n4; i4 += 2 * stride) {
        int32_t c4b = c4, hb = h;
        advance(c4b, hb);
        const float4 x0 = load4(f, i4 * 4);
        const float4 x1 = load4(f, (i4 + stride) * 4);
        const float lam0 = -expf(__ldg(A_log + h)), lam1 = -expf(__ldg(A_log + hb));
        const float4 d0 = __ldg(reinterpret_cast<const float4*>(dt_bias + (int64_t)h * K + 4 * c4));
        const float4 d1 = __ldg(reinterpret_cast<const float4*>(dt_bias + (int64_t)hb * K + 4 * c4b));
        float4 r0, r1;
        r0.x = gate_decay(x0.x, d0.x, lam0);
        r0.y = gate_decay(x0.y, d0.y, lam0);
        r0.z = gate_decay(x0.z, d0.z, lam0);
        r0.w = gate_decay(x0.w, d0.w, lam0);
        r1.x = gate_decay(x1.x, d1.x, lam1);
        r1.y = gate_decay(x1.y, d1.y, lam1);
        r1.z = gate_decay(x1.z, d1.z, lam1);
        r1.w = gate_decay(x1.w, d1.w, lam1);
        __stcs(reinterpret_cast<float4*>(g_out + i4 * 4), r0);
        __stcs(reinterpret_cast<float4*>(g_out + (i4 + stride) * 4), r1);
        c4 = c4b;
        h = hb;
        advance(c4, h);
    }
    if (i4 < n4) decay4(i4, c4, h);
    const int64_t nb = T * H;
    for (int64_t i = start; i < nb; i += stride) {
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
