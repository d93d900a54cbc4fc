// kda_recurrent_step: one token of the KDA recurrence per sequence (decode).
//
//   S <- (I - beta k^ k^^T) Diag(e^g) S + beta k^ v^T,   o = scale * S^T q^
//
// The token-by-token FP32 recurrence is the serving-side path the pages
// compare the chunked kernel against ("Add opt-in FP32 KDA chunk
// computation", section Problem).  One 256-thread CTA per (sequence, head);
// the two adjacent lanes 2v, 2v+1 keep rows 0-63 and 64-127 of column v of S
// in registers, so the decay, S^T k^, the rank-1 write and S^T q^ need only
// one shuffle between the two lanes; q^, k^ and e^g are shared.
// HBM-bound: 2 K V 4 bytes of state read and written per (sequence, head).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int DK = kHeadK;
constexpr int DV = kHeadV;
constexpr int NT = 256;
constexpr int RH = DK / 2;   // rows of S per thread

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NT) recurrent_step_kernel(StepArgs a)
{
    __shared__ float qs[DK], ks[DK], as[DK];
    __shared__ float red[2][DK / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int col = t >> 1, hf = t & 1, c0 = RH * hf;
    const int64_t unit = blockIdx.x;                    // n * H + h
    const TIn* q = static_cast<const TIn*>(a.q) + unit * DK;
    const TIn* k = static_cast<const TIn*>(a.k) + unit * DK;
    const TIn* v = static_cast<const TIn*>(a.v) + unit * DV;
    float* st = a.state + unit * DK * DV;

    float S[RH];
#pragma unroll
    for (int c = 0; c < RH; ++c) S[c] = st[(int64_t)(c0 + c) * DV + col];
    const float vv = load_as_float(v + col);
    const float beta = a.beta[unit];

    if (t < DK) {
        const float qv = load_as_float(q + t), kv = load_as_float(k + t);
        float sq = qv * qv, sk = kv * kv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        if (lane == 0) {
            red[0][warp] = sq;
            red[1][warp] = sk;
        }
        qs[t] = qv;
        ks[t] = kv;
        as[t] = expf(a.g[unit * DK + t]);
    }
    __syncthreads();
    float tq = 0.f, tk = 0.f;
#pragma unroll
    for (int w = 0; w < DK / 32; ++w) {
        tq += red[0][w];
        tk += red[1][w];
    }
    const float iq = a.l2norm ? 1.f / sqrtf(tq + 1e-6f) : 1.f;
    const float ik = a.l2norm ? 1.f / sqrtf(tk + 1e-6f) : 1.f;

    float r = 0.f;
#pragma unroll
    for (int c = 0; c < RH; ++c) {
        S[c] *= as[c0 + c];
        r += S[c] * ks[c0 + c];
    }
    r = ik * (r + __shfl_xor_sync(0xffffffffu, r, 1));  // S^T k^ over all 128 rows
    const float w = beta * (vv - r) * ik;                // the write uses k^ = ik k
    float o = 0.f;
#pragma unroll
    for (int c = 0; c < RH; ++c) {
        S[c] += ks[c0 + c] * w;
        o += S[c] * qs[c0 + c];
    }
    o = iq * (o + __shfl_xor_sync(0xffffffffu, o, 1));
    if (hf == 0) store_out(static_cast<TOut*>(a.out) + unit * DV + col, a.scale * o);
#pragma unroll
    for (int c = 0; c < RH; ++c) st[(int64_t)(c0 + c) * DV + col] = S[c];
}

template <typename TIn, typename TOut>
cudaError_t launch_typed(const StepArgs& a, cudaStream_t stream)
{
    const int64_t units = (int64_t)a.N * a.H;
    if (units > INT32_MAX) return cudaErrorInvalidConfiguration;
    recurrent_step_kernel<TIn, TOut><<<(unsigned)units, NT, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent_step(const StepArgs& a, cudaStream_t stream)
{
    if (a.qkv_bf16)
        return a.out_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(a, stream)
                          : launch_typed<__nv_bfloat16, float>(a, stream);
    return a.out_bf16 ? launch_typed<float, __nv_bfloat16>(a, stream)
                      : launch_typed<float, float>(a, stream);
}

}  // namespace kda
