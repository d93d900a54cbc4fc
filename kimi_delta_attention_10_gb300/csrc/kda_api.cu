// Host side of the C ABI declared in include/kda.h: argument validation and
// dispatch.  Nothing is launched unless every host-visible check passes.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "kda.h"
#include "kda_internal.cuh"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_dtype(int32_t d) { return d == KDA_F32 || d == KDA_BF16; }

// kda_test_set_fault's setting, read by every chunk-forward launch.
std::atomic<int32_t> g_test_fault{KDA_TEST_FAULT_NONE};

}  // namespace

namespace kda {

int32_t test_fault() { return g_test_fault.load(std::memory_order_relaxed); }

int device_sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace kda

extern "C" {

int32_t kda_abi_version(void) { return 3; }

const char* kda_status_string(int32_t s)
{
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported shape, dtype or mode";
        case KDA_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_TIMEOUT: return "device wait timed out";
        case KDA_ERR_DEVICE_ARG: return "device saw offsets outside [0, T]";
        case KDA_ERR_TOO_LARGE:
            return "problem needs more than the 64 MiB static scratch of kda_chunk_fwd_static";
        case KDA_ERR_RANGE:
            return "device stored a non-finite value (an input or an FP16 operand out of range)";
        default: return "unknown status";
    }
}

kda_status kda_gate(const void* f, int32_t f_dtype, const float* A_log, const float* dt_bias,
                    const void* b, int32_t b_dtype, int64_t T, int32_t H, int32_t K,
                    float* g_out, float* beta_out, kda_stream_t stream)
{
    if (T < 0 || H < 1 || K < 1) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(f_dtype) || !valid_dtype(b_dtype)) return KDA_ERR_INVALID_ARG;
    if (K % 4 != 0) return KDA_ERR_UNSUPPORTED;
    if (T == 0) return KDA_OK;   // nothing to do; empty tensors may have NULL data
    if (!f || !A_log || !dt_bias || !b || !g_out || !beta_out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(f) || !aligned16(A_log) || !aligned16(dt_bias) || !aligned16(b) ||
        !aligned16(g_out) || !aligned16(beta_out))
        return KDA_ERR_ALIGNMENT;
    cudaError_t e = kda::launch_gate(f, f_dtype == KDA_BF16, A_log, dt_bias, b,
                                     b_dtype == KDA_BF16, T, H, K, g_out, beta_out,
                                     reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

namespace {

// Shared validation of the chunk entry points (everything but g/beta vs the
// gate inputs).  Returns KDA_OK when a launch may proceed.
kda_status check_chunk(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                       const int32_t* cu_seqlens, const int32_t* cu_seqlens_host, int32_t N,
                       int64_t T, int32_t H, int32_t K, int32_t V, int32_t qk_l2norm,
                       int32_t mode, const void* out, int32_t out_dtype,
                       const float* initial_state, const float* final_state,
                       const int32_t* status_dev)
{
    if (N < 0 || T < 0 || H < 1 || K < 1 || V < 1) return KDA_ERR_INVALID_ARG;
    if (T > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (!valid_dtype(qkv_dtype) || !valid_dtype(out_dtype)) return KDA_ERR_INVALID_ARG;
    if (mode != KDA_MODE_BF16_TC && mode != KDA_MODE_FP32_EXACT) return KDA_ERR_INVALID_ARG;
    if (qk_l2norm != 0 && qk_l2norm != 1) return KDA_ERR_INVALID_ARG;
    if (K != kda::kHeadK || V != kda::kHeadV) return KDA_ERR_UNSUPPORTED;
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !out)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, cu_seqlens, out, initial_state, final_state, status_dev};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || (int64_t)cu_seqlens_host[N] != T)
            return KDA_ERR_INVALID_ARG;
        for (int32_t n = 0; n < N; ++n)
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

// Workspace checks and dispatch.
kda_status launch_chunk(kda::ChunkArgs a, int32_t mode, const int32_t* cu_seqlens_host,
                        void* workspace, int64_t workspace_bytes, kda_stream_t stream,
                        bool overlap = true)
{
    const bool split = mode == KDA_MODE_BF16_TC && workspace != nullptr;
    if (split) {
        if (!aligned16(workspace)) return KDA_ERR_ALIGNMENT;
        if (workspace_bytes < kda::split_workspace_bytes(a.N, a.T, a.H)) return KDA_ERR_INVALID_ARG;
    }
    // FP32-exact mode runs in two phases when its workspace fits, else in the
    // single-pass kernel (a smaller workspace is not used)
    const bool split32 = mode == KDA_MODE_FP32_EXACT && workspace != nullptr &&
                         workspace_bytes >= kda::fp32_split_workspace_bytes(a.N, a.T, a.H);
    if (split32 && !aligned16(workspace)) return KDA_ERR_ALIGNMENT;
    if (a.N == 0) return KDA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (split || split32) {
        a.workspace = workspace;
        int64_t chunks = kda::split_chunk_bound(a.N, a.T);
        if (cu_seqlens_host) {            // exact count: no idle preparation CTAs
            chunks = 0;
            for (int32_t n = 0; n < a.N; ++n)
                chunks += (cu_seqlens_host[n + 1] - cu_seqlens_host[n] + kda::kChunk - 1) / kda::kChunk;
        }
        e = split ? kda::launch_chunk_split(a, chunks, overlap, s)
                  : kda::launch_chunk_fp32_split(a, chunks, s);
    } else {
        e = (mode == KDA_MODE_BF16_TC) ? kda::launch_chunk_tc(a, s) : kda::launch_chunk_fp32(a, s);
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda::ChunkArgs chunk_args(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                          const int32_t* cu_seqlens, int32_t N, int64_t T, int32_t H,
                          float scale, int32_t qk_l2norm, void* out, int32_t out_dtype,
                          const float* initial_state, float* final_state, int32_t* status_dev)
{
    kda::ChunkArgs a = {};
    a.q = q; a.k = k; a.v = v; a.cu_seqlens = cu_seqlens;
    a.N = N; a.T = T; a.H = H; a.scale = scale; a.l2norm = qk_l2norm;
    a.out = out; a.final_state = final_state; a.status = status_dev;
    a.qkv_bf16 = qkv_dtype == KDA_BF16; a.out_bf16 = out_dtype == KDA_BF16;
    a.initial_state = initial_state;
    a.fault = kda::test_fault();
    return a;
}

}  // namespace

kda_status kda_chunk_workspace_size(int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                                    int32_t mode, int64_t* bytes_host)
{
    if (!bytes_host) return KDA_ERR_INVALID_ARG;
    if (N < 0 || T < 0 || H < 1 || K < 1 || V < 1) return KDA_ERR_INVALID_ARG;
    if (mode != KDA_MODE_BF16_TC && mode != KDA_MODE_FP32_EXACT) return KDA_ERR_INVALID_ARG;
    if (T > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (K != kda::kHeadK || V != kda::kHeadV) return KDA_ERR_UNSUPPORTED;
    *bytes_host = mode == KDA_MODE_BF16_TC ? kda::split_workspace_bytes(N, T, H)
                                           : kda::fp32_split_workspace_bytes(N, T, H);
    return KDA_OK;
}

kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                         const float* g, const float* beta,
                         const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                         int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                         float scale, int32_t qk_l2norm, int32_t mode,
                         void* out, int32_t out_dtype, const float* initial_state,
                         float* final_state, void* workspace, int64_t workspace_bytes,
                         int32_t* status_dev, kda_stream_t stream)
{
    kda_status st = check_chunk(q, k, v, qkv_dtype, cu_seqlens, cu_seqlens_host, N, T, H, K, V,
                                qk_l2norm, mode, out, out_dtype, initial_state, final_state,
                                status_dev);
    if (st != KDA_OK) return st;
    if (T > 0 && (!g || !beta)) return KDA_ERR_INVALID_ARG;
    if ((g && !aligned16(g)) || (beta && !aligned16(beta))) return KDA_ERR_ALIGNMENT;
    kda::ChunkArgs a = chunk_args(q, k, v, qkv_dtype, cu_seqlens, N, T, H, scale, qk_l2norm, out,
                                  out_dtype, initial_state, final_state, status_dev);
    a.g = g; a.beta = beta; a.gated = false;
    return launch_chunk(a, mode, cu_seqlens_host, workspace, workspace_bytes, stream);
}

kda_status kda_chunk_fwd_gated(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                               const void* f, int32_t f_dtype, const float* A_log,
                               const float* dt_bias, const void* b, int32_t b_dtype,
                               const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                               int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                               float scale, int32_t qk_l2norm, int32_t mode,
                               void* out, int32_t out_dtype, const float* initial_state,
                               float* final_state, void* workspace, int64_t workspace_bytes,
                               int32_t* status_dev, kda_stream_t stream)
{
    kda_status st = check_chunk(q, k, v, qkv_dtype, cu_seqlens, cu_seqlens_host, N, T, H, K, V,
                                qk_l2norm, mode, out, out_dtype, initial_state, final_state,
                                status_dev);
    if (st != KDA_OK) return st;
    if (!valid_dtype(f_dtype) || !valid_dtype(b_dtype)) return KDA_ERR_INVALID_ARG;
    if (!A_log || !dt_bias) return KDA_ERR_INVALID_ARG;
    if (T > 0 && (!f || !b)) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {f, A_log, dt_bias, b};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGNMENT;
    kda::ChunkArgs a = chunk_args(q, k, v, qkv_dtype, cu_seqlens, N, T, H, scale, qk_l2norm, out,
                                  out_dtype, initial_state, final_state, status_dev);
    a.gated = true;
    a.f = f;
    a.f_bf16 = f_dtype == KDA_BF16;
    a.A_log = A_log;
    a.dt_bias = dt_bias;
    a.b = b;
    a.b_bf16 = b_dtype == KDA_BF16;
    return launch_chunk(a, mode, cu_seqlens_host, workspace, workspace_bytes, stream);
}

kda_status kda_chunk_fwd_gated_norm(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                                    const void* f, int32_t f_dtype, const float* A_log,
                                    const float* dt_bias, const void* b, int32_t b_dtype,
                                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                    int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                                    float scale, int32_t qk_l2norm, int32_t mode,
                                    const void* z, int32_t z_dtype, const float* weight,
                                    float eps, void* out, int32_t out_dtype,
                                    const float* initial_state, float* final_state,
                                    void* workspace, int64_t workspace_bytes,
                                    int32_t* status_dev, kda_stream_t stream)
{
    kda_status st = check_chunk(q, k, v, qkv_dtype, cu_seqlens, cu_seqlens_host, N, T, H, K, V,
                                qk_l2norm, mode, out, out_dtype, initial_state, final_state,
                                status_dev);
    if (st != KDA_OK) return st;
    if (!valid_dtype(f_dtype) || !valid_dtype(b_dtype) || !valid_dtype(z_dtype))
        return KDA_ERR_INVALID_ARG;
    if (!A_log || !dt_bias || !weight || !(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
    if (T > 0 && (!f || !b || !z)) return KDA_ERR_INVALID_ARG;
    if (z != nullptr && z == out) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {f, A_log, dt_bias, b, z, weight};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGNMENT;
    kda::ChunkArgs a = chunk_args(q, k, v, qkv_dtype, cu_seqlens, N, T, H, scale, qk_l2norm, out,
                                  out_dtype, initial_state, final_state, status_dev);
    a.gated = true;
    a.f = f;
    a.f_bf16 = f_dtype == KDA_BF16;
    a.A_log = A_log;
    a.dt_bias = dt_bias;
    a.b = b;
    a.b_bf16 = b_dtype == KDA_BF16;
    if (mode == KDA_MODE_BF16_TC && workspace != nullptr && z_dtype == KDA_BF16) {
        // fused: the scan stores y in place of o
        a.out_norm = true;
        a.z = static_cast<const __nv_bfloat16*>(z);
        a.norm_w = weight;
        a.norm_eps = eps;
        return launch_chunk(a, mode, cu_seqlens_host, workspace, workspace_bytes, stream);
    }
    st = launch_chunk(a, mode, cu_seqlens_host, workspace, workspace_bytes, stream);
    if (st != KDA_OK || N == 0 || T == 0) return st;
    cudaError_t e = kda::launch_gated_rmsnorm(out, out_dtype == KDA_BF16, z, z_dtype == KDA_BF16,
                                              weight, T * H, eps, out, out_dtype == KDA_BF16,
                                              reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_chunk_fwd_static(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                                const float* g, const float* beta,
                                const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                                float scale, int32_t qk_l2norm, void* out, int32_t out_dtype,
                                const float* initial_state, float* final_state,
                                int32_t* status_dev, kda_stream_t stream)
{
    kda_status st = check_chunk(q, k, v, qkv_dtype, cu_seqlens, cu_seqlens_host, N, T, H, K, V,
                                qk_l2norm, KDA_MODE_BF16_TC, out, out_dtype, initial_state,
                                final_state, status_dev);
    if (st != KDA_OK) return st;
    if (T > 0 && (!g || !beta)) return KDA_ERR_INVALID_ARG;
    if ((g && !aligned16(g)) || (beta && !aligned16(beta))) return KDA_ERR_ALIGNMENT;
    if (kda::split_workspace_bytes(N, T, H) > kda::kStaticScratchBytes) return KDA_ERR_TOO_LARGE;
    if (N == 0) return KDA_OK;
    {
        // the scratch address is the current device's: the stream must be on it
        int cur = 0, sdev = 0;
        if (cudaGetDevice(&cur) != cudaSuccess) return KDA_ERR_CUDA;
        if (cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (sdev != cur) return KDA_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    if (kda::static_scratch(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    kda::ChunkArgs a = chunk_args(q, k, v, qkv_dtype, cu_seqlens, N, T, H, scale, qk_l2norm, out,
                                  out_dtype, initial_state, final_state, status_dev);
    a.g = g; a.beta = beta; a.gated = false;
    // one window: the schedule the bit-for-bit tests compare the windows with
    return launch_chunk(a, KDA_MODE_BF16_TC, cu_seqlens_host, scratch, kda::kStaticScratchBytes,
                        stream, false);
}

kda_status kda_recurrent_step(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                              const float* g, const float* beta, int32_t N, int32_t H,
                              int32_t K, int32_t V, float scale, int32_t qk_l2norm,
                              float* state, void* out, int32_t out_dtype,
                              kda_stream_t stream)
{
    if (N < 0 || H < 1 || K < 1 || V < 1) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(qkv_dtype) || !valid_dtype(out_dtype)) return KDA_ERR_INVALID_ARG;
    if (qk_l2norm != 0 && qk_l2norm != 1) return KDA_ERR_INVALID_ARG;
    if (K != kda::kHeadK || V != kda::kHeadV) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, g, beta, state, out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
    kda::StepArgs a = {};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.N = N; a.H = H; a.scale = scale;
    a.l2norm = qk_l2norm; a.state = state; a.out = out;
    a.qkv_bf16 = qkv_dtype == KDA_BF16; a.out_bf16 = out_dtype == KDA_BF16;
    cudaError_t e = kda::launch_recurrent_step(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_gated_rmsnorm(const void* o, int32_t o_dtype, const void* z, int32_t z_dtype,
                             const float* weight, int64_t rows, int32_t V, float eps, void* y,
                             int32_t y_dtype, kda_stream_t stream)
{
    if (rows < 0 || V < 1 || !(eps >= 0.f)) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(o_dtype) || !valid_dtype(z_dtype) || !valid_dtype(y_dtype))
        return KDA_ERR_INVALID_ARG;
    if (V != kda::kHeadV) return KDA_ERR_UNSUPPORTED;
    if (rows == 0) return KDA_OK;
    if (!o || !z || !weight || !y) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {o, z, weight, y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (y == o && y_dtype != o_dtype) return KDA_ERR_INVALID_ARG;
    cudaError_t e = kda::launch_gated_rmsnorm(o, o_dtype == KDA_BF16, z, z_dtype == KDA_BF16,
                                              weight, rows, eps, y, y_dtype == KDA_BF16,
                                              reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_chunk_bwd_workspace_size(int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                                        int64_t* bytes_host)
{
    if (!bytes_host) return KDA_ERR_INVALID_ARG;
    if (N < 0 || T < 0 || H < 1 || K < 1 || V < 1) return KDA_ERR_INVALID_ARG;
    if (T > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (K != kda::kHeadK || V != kda::kHeadV) return KDA_ERR_UNSUPPORTED;
    *bytes_host = kda::bwd_workspace_bytes(N, T, H);
    return KDA_OK;
}

kda_status kda_chunk_bwd(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                         const float* g, const float* beta,
                         const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                         int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                         float scale, int32_t qk_l2norm,
                         const void* dout, int32_t dout_dtype,
                         const float* initial_state, const float* dfinal_state,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta,
                         float* dinitial_state, void* workspace, int64_t workspace_bytes,
                         int32_t* status_dev, kda_stream_t stream)
{
    kda_status st = check_chunk(q, k, v, qkv_dtype, cu_seqlens, cu_seqlens_host, N, T, H, K, V,
                                qk_l2norm, KDA_MODE_FP32_EXACT, dout, dout_dtype, initial_state,
                                dfinal_state, status_dev);
    if (st != KDA_OK) return st;
    if (T > 0 && (!g || !beta || !dq || !dk || !dv || !dg || !dbeta)) return KDA_ERR_INVALID_ARG;
    if (N > 0 && !workspace) return KDA_ERR_INVALID_ARG;
    const void* ptrs[] = {g, beta, dq, dk, dv, dg, dbeta, dinitial_state, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_ALIGNMENT;
    if (N > 0 && workspace_bytes < kda::bwd_workspace_bytes(N, T, H)) return KDA_ERR_INVALID_ARG;
    // no output may be an input or another output (checked on the base pointers)
    const void* outs[] = {dq, dk, dv, dg, dbeta, dinitial_state};
    const void* ins[] = {q, k, v, g, beta, dout, initial_state, dfinal_state, cu_seqlens, workspace};
    for (int i = 0; i < 6; ++i) {
        if (!outs[i]) continue;
        for (const void* p : ins)
            if (p == outs[i]) return KDA_ERR_INVALID_ARG;
        for (int j = i + 1; j < 6; ++j)
            if (outs[j] == outs[i]) return KDA_ERR_INVALID_ARG;
    }
    if (N == 0) return KDA_OK;
    kda::BwdLaunch a = {};
    a.q = q; a.k = k; a.v = v; a.qkv_bf16 = qkv_dtype == KDA_BF16; a.g = g; a.beta = beta;
    a.cu = cu_seqlens; a.N = N; a.T = T; a.H = H; a.scale = scale; a.l2norm = qk_l2norm;
    a.dout = dout; a.dout_bf16 = dout_dtype == KDA_BF16;
    a.init = initial_state; a.dfinal = dfinal_state;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dinit = dinitial_state;
    a.workspace = workspace; a.status = status_dev;
    cudaError_t e = kda::launch_chunk_bwd(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_test_set_fault(int32_t where)
{
    if (where < KDA_TEST_FAULT_NONE || where > KDA_TEST_FAULT_SINGLE_PASS)
        return KDA_ERR_INVALID_ARG;
    g_test_fault.store(where, std::memory_order_relaxed);
    return KDA_OK;
}

}  // extern "C"
