// Internal declarations shared by the library's translation units (not public).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;     // tokens per chunk
constexpr int kHeadK = 128;    // supported key dim
constexpr int kHeadV = 128;    // supported value dim

struct ChunkArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu_seqlens;
    int32_t N;
    int64_t T;
    int32_t H;
    float scale;
    int32_t l2norm;
    void* out;
    float* final_state;
    int32_t* status;
    bool qkv_bf16;
    bool out_bf16;
};

// Each launcher returns cudaSuccess or the launch error.
cudaError_t launch_gate(const void* f, bool f_bf16, const float* A_log, const float* dt_bias,
                        const void* b, bool b_bf16, int64_t T, int32_t H, int32_t K,
                        float* g_out, float* beta_out, cudaStream_t stream);

cudaError_t launch_chunk_fp32(const ChunkArgs& a, cudaStream_t stream);
cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t stream);

int device_sm_count();

// Records the first device-side error in the caller's status word.
__device__ __forceinline__ void report_status(int32_t* status, int32_t code)
{
    if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float load_as_float(const float* p) { return *p; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16* p)
{
    return __bfloat162float(*p);
}

}  // namespace kda
