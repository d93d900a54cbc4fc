// kda_gated_rmsnorm: the KDA output gate with gated RMSNorm, per (token, head)
// row of V values:
//     y = o / sqrt(mean(o^2) + eps) * w * sigmoid(z)
// (the low-rank output gate and "gated-norm" of "GLM-5.3-Flash F6.2: KDA
// correctness and FLA sequence parallelism", module and FLA-SP commits; the
// pages print no formula, this is its plain reading).
//
// HBM-bound: one warp per row of 128, four values per lane (one 8- or 16-byte
// load of o and of z, one store of y), the sum of squares reduced by shuffles;
// each warp keeps two rows' loads in flight, grid-stride.  Algorithmic bytes per row:
// V * (sizeof o + sizeof z + sizeof y).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

__device__ __forceinline__ float4 load4v(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4v(const __nv_bfloat16* p)
{
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ void store4v(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void store4v(__nv_bfloat16* p, float4 v)
{
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}

template <typename TO, typename TZ, typename TY>
__global__ void __launch_bounds__(256) gated_rmsnorm_kernel(const TO* __restrict__ o,
                                                            const TZ* __restrict__ z,
                                                            const float* __restrict__ w,
                                                            int64_t rows, float eps,
                                                            TY* __restrict__ y)
{
    constexpr int V = kHeadV;
    constexpr int kRows = 2;                       // rows in flight per warp
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const float4 wv = __ldg(reinterpret_cast<const float4*>(w) + lane);
    for (int64_t r0 = warp0; r0 < rows; r0 += kRows * nwarps) {
        int64_t rr[kRows];
#pragma unroll
        for (int k = 0; k < kRows; ++k) rr[k] = r0 + k * nwarps;
        float4 ov[kRows], zv[kRows];
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            if (rr[k] < rows) {
                ov[k] = load4v(o + rr[k] * V + 4 * lane);
                zv[k] = load4v(z + rr[k] * V + 4 * lane);
            }
        }
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            if (rr[k] >= rows) break;              // warp-uniform
            float ss = ov[k].x * ov[k].x + ov[k].y * ov[k].y + ov[k].z * ov[k].z + ov[k].w * ov[k].w;
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            const float inv = 1.f / sqrtf(ss * (1.f / V) + eps);
            float4 res;
            res.x = ov[k].x * inv * wv.x * gate_sigmoid(zv[k].x);
            res.y = ov[k].y * inv * wv.y * gate_sigmoid(zv[k].y);
            res.z = ov[k].z * inv * wv.z * gate_sigmoid(zv[k].z);
            res.w = ov[k].w * inv * wv.w * gate_sigmoid(zv[k].w);
            store4v(y + rr[k] * V + 4 * lane, res);
        }
    }
}

template <typename TO, typename TZ, typename TY>
cudaError_t launch_typed(const void* o, const void* z, const float* w, int64_t rows, float eps,
                         void* y, cudaStream_t stream)
{
    const int sms = device_sm_count();
    const int64_t max_blocks = (int64_t)(sms > 0 ? sms : 152) * 8;   // 8 x 256 threads per SM
    int64_t blocks = (rows + 15) / 16;            // 8 warps x 2 rows per block
    if (blocks > max_blocks) blocks = max_blocks;
    if (blocks < 1) blocks = 1;
    gated_rmsnorm_kernel<TO, TZ, TY><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const TO*>(o), static_cast<const TZ*>(z), w, rows, eps, static_cast<TY*>(y));
    return cudaGetLastError();
}

template <typename TO, typename TZ>
cudaError_t launch_y(const void* o, const void* z, const float* w, int64_t rows, float eps,
                     void* y, bool y_bf16, cudaStream_t stream)
{
    return y_bf16 ? launch_typed<TO, TZ, __nv_bfloat16>(o, z, w, rows, eps, y, stream)
                  : launch_typed<TO, TZ, float>(o, z, w, rows, eps, y, stream);
}

template <typename TO>
cudaError_t launch_z(const void* o, const void* z, bool z_bf16, const float* w, int64_t rows,
                     float eps, void* y, bool y_bf16, cudaStream_t stream)
{
    return z_bf16 ? launch_y<TO, __nv_bfloat16>(o, z, w, rows, eps, y, y_bf16, stream)
                  : launch_y<TO, float>(o, z, w, rows, eps, y, y_bf16, stream);
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const void* o, bool o_bf16, const void* z, bool z_bf16,
                                 const float* w, int64_t rows, float eps, void* y, bool y_bf16,
                                 cudaStream_t stream)
{
    return o_bf16 ? launch_z<__nv_bfloat16>(o, z, z_bf16, w, rows, eps, y, y_bf16, stream)
                  : launch_z<float>(o, z, z_bf16, w, rows, eps, y, y_bf16, stream);
}

}  // namespace kda
