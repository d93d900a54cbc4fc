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
    const float* initial_state;   // [N,H,K,V] or nullptr
    // Gate fused into the prologue (kda_chunk_fwd_gated): g and beta are then
    // formed from f, A_log, dt_bias and b, and the g/beta pointers are unused.
    bool gated;
    const void* f;                // [T,H,K] F32 or BF16 (f_bf16)
    bool f_bf16;
    const float* A_log;
    const float* dt_bias;
    const void* b;
    bool b_bf16;
    // Two-phase tensor-core path: caller-provided scratch of at least
    // split_workspace_bytes(N, T, H) bytes (nullptr: single-pass kernel).
    void* workspace;
    // Output gate fused into the scan's output store (kda_chunk_fwd_gated_norm,
    // two-phase path, BF16 z): out receives
    //   y = o / sqrt(mean_v o^2 + norm_eps) * norm_w[v] * sigmoid(z)
    // instead of o.
    bool out_norm;
    const __nv_bfloat16* z;       // [T,H,V]
    const float* norm_w;          // [V]
    float norm_eps;
    // Test hook (kda_test_set_fault): a KDA_TEST_FAULT_* value; the named
    // kernel's CTA 0 withholds one arrival so that its bounded wait gives up.
    int32_t fault;
};

// The current test-hook setting (0 unless a test set one).
int32_t test_fault();

// Where a chunk kernel's decay comes from: g given (kda_chunk_fwd), or formed
// from the gate's pre-activation f read as F32 or as BF16 (kda_chunk_fwd_gated).
enum GateIn : int { kGateG = 0, kGateF32 = 1, kGateBF16 = 2 };
template <int kGate> struct GateSrc { using T = float; };
template <> struct GateSrc<kGateBF16> { using T = __nv_bfloat16; };

// The decay input of a launch: the pointer and the GateIn value it needs.
inline int gate_in(const ChunkArgs& a) { return !a.gated ? kGateG : a.f_bf16 ? kGateBF16 : kGateF32; }

struct StepArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    int32_t N;
    int32_t H;
    float scale;
    int32_t l2norm;
    float* state;
    void* out;
    bool qkv_bf16;
    bool out_bf16;
};

// Each launcher returns cudaSuccess or the launch error.
cudaError_t launch_gate(const void* f, bool f_bf16, const float* A_log, const float* dt_bias,
                        const void* b, bool b_bf16, int64_t T, int32_t H, int32_t K,
                        float* g_out, float* beta_out, cudaStream_t stream);

cudaError_t launch_chunk_fp32(const ChunkArgs& a, cudaStream_t stream);
cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t stream);
// Two-phase path; `chunks` bounds the number of chunks over all sequences.
// `overlap` lets the preparation of later chunks run beside the scan of
// earlier ones (chunk windows; programmatic dependent launch on `stream`).
cudaError_t launch_chunk_split(const ChunkArgs& a, int64_t chunks, bool overlap,
                               cudaStream_t stream);
// Chunks of N packed sequences of T tokens in all, at most.
__host__ __device__ inline int64_t split_chunk_bound(int32_t N, int64_t T) { return T / kChunk + N; }
// The plan kernel: int32 header with [0] = bad-offsets flag and, from
// [kPlanOffsets], the per-sequence chunk offsets (N + 1 of them).
constexpr int kPlanOffsets = 4;
int64_t chunk_plan_header_bytes(int32_t N);
cudaError_t launch_chunk_plan(const int32_t* cu, int32_t N, int64_t T, int32_t* hdr,
                              int32_t* status, cudaStream_t stream);
int64_t split_workspace_bytes(int32_t N, int64_t T, int32_t H);
// FP32-exact mode in two phases (kda_chunk_fp32_split.cu): plan header and one
// FP32 record per (chunk bound, head).
int64_t fp32_split_workspace_bytes(int32_t N, int64_t T, int32_t H);
cudaError_t launch_chunk_fp32_split(const ChunkArgs& a, int64_t chunks, cudaStream_t stream);
// The static scratch of kda_chunk_fwd_static and its size; static_scratch()
// returns its address on the current device (looked up once per device).
constexpr int64_t kStaticScratchBytes = 64ll << 20;
cudaError_t static_scratch(void** ptr);
cudaError_t launch_recurrent_step(const StepArgs& a, cudaStream_t stream);
cudaError_t launch_gated_rmsnorm(const void* o, bool o_bf16, const void* z, bool z_bf16,
                                 const float* w, int64_t rows, float eps, void* y, bool y_bf16,
                                 cudaStream_t stream);

// Backward (kda_chunk_bwd): FP32 outputs, workspace of bwd_workspace_bytes.
struct BwdLaunch {
    const void* q;
    const void* k;
    const void* v;
    bool qkv_bf16;
    const float* g;
    const float* beta;
    const int32_t* cu;
    int32_t N;
    int64_t T;
    int32_t H;
    float scale;
    int32_t l2norm;
    const void* dout;
    bool dout_bf16;
    const float* init;     // [N,H,K,V] or nullptr
    const float* dfinal;   // [N,H,K,V] or nullptr
    float* dq;
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    float* dinit;          // or nullptr
    void* workspace;
    int32_t* status;
};
int64_t bwd_workspace_bytes(int32_t N, int64_t T, int32_t H);
cudaError_t launch_chunk_bwd(const BwdLaunch& a, cudaStream_t stream);

int device_sm_count();

// Records the first device-side error in the caller's status word.
__device__ __forceinline__ void report_status(int32_t* status, int32_t code)
{
    if (status != nullptr) atomicCAS(status, 0, code);
}

// The gate's FP32 arithmetic, shared by kda_gate and the fused prologues so
// that both give identical values: g = lamneg * softplus(x), lamneg = -exp(A_log).
// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(y), y = e^{-|x|} in (0, 1].
// log1p(y) = 2 atanh(s) with s = y / (2 + y) in (0, 1/3], and atanh(s) is the
// odd series s + s^3/3 + s^5/5 + ...; eight terms leave a truncation below
// s^17/17 < 2e-9 relative.  The quotient uses the fast (2-ulp) division.
// Measured against FP64 over x in [-40, 20): max relative error 2.7e-7.
__device__ __forceinline__ float gate_softplus(float x)
{
    const float y = expf(-fabsf(x));
    const float s = __fdividef(y, 2.f + y);
    const float z = s * s;
    float p = 1.f / 17.f;
    p = fmaf(p, z, 1.f / 15.f);
    p = fmaf(p, z, 1.f / 13.f);
    p = fmaf(p, z, 1.f / 11.f);
    p = fmaf(p, z, 1.f / 9.f);
    p = fmaf(p, z, 1.f / 7.f);
    p = fmaf(p, z, 1.f / 5.f);
    p = fmaf(p, z, 1.f / 3.f);
    return fmaxf(x, 0.f) + 2.f * fmaf(s * z, p, s);
}
__device__ __forceinline__ float gate_sigmoid(float x) { return 1.f / (1.f + expf(-x)); }
// g from its pre-activation f, dt_bias and lamneg = -exp(A_log[h]); the explicit
// roundings keep the product from being contracted into a later expf.
__device__ __forceinline__ float gate_decay(float f, float dt_bias, float lamneg)
{
    return __fmul_rn(lamneg, gate_softplus(__fadd_rn(f, dt_bias)));
}

// e^g for g = lamneg * softplus(f + dt_bias), formed directly for the tensor-core
// path: e^g = (1 + e^x)^lamneg = 2^(lamneg * log2(1 + 2^(x log2 e))), three
// hardware ex2/lg2 approximations instead of the accurate softplus and exp.
// Its relative error stays below 1e-5 wherever e^g is above FP16's smallest
// subnormal (a float32 model with the instructions' error bounds gives 8.6e-6
// at exp(A_log) = 16 and 3e-7 at 0.05), 50 times below the 2^-11 rounding of
// the FP16 operands it feeds.  For x below -17, 1 + e^x rounds to 1 and e^g to
// 1 (true value within 1e-6 of it); for x above 88, e^x overflows and e^g is
// 0, its limit.  The FP32-exact path keeps gate_decay.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float gate_exp_fast(float f, float dt_bias, float lamneg)
{
    const float e = ex2_approx((f + dt_bias) * 1.4426950408889634f);
    return ex2_approx(lamneg * lg2_approx(1.f + e));
}

__device__ __forceinline__ float load_as_float(const float* p) { return *p; }
__device__ __forceinline__ float load_as_float(const __nv_bfloat16* p)
{
    return __bfloat162float(*p);
}

}  // namespace kda
