// kda_chunk_bwd: the vector-Jacobian product of the KDA forward, IEEE FP32.
//
// The backward of the chunked forward (tested against FP64 budgets in "Add
// opt-in FP32 KDA chunk computation", section Validation) is the VJP of the
// token recurrence (per sequence and head, q^ and k^ L2-normalised):
//   S'_t = Diag(e^{g_t}) S_{t-1},  u_t = S'_t^T k^_t,  d_t = beta_t (v_t - u_t),
//   S_t  = S'_t + k^_t d_t^T,      o_t = scale S_t^T q^_t.
// Walking the tokens backwards with dS (the gradient of the state):
//   dS += scale q^_t dO_t^T;  dq^_t = scale S_t dO_t
//   dd = dS^T k^_t;  dv_t = beta dd;  du = -beta dd;  dbeta_t = dd . (v_t - u_t)
//   dk^_t = dS d_t + S'_t du;  dS' = dS + k^_t du^T
//   dg_t = rowsum(dS' o S'_t);  dS <- Diag(e^{g_t}) dS'
// then dq = (dq^ - q^ (q^ . dq^)) / n for n = sqrt(|q|^2 + eps) (k alike).
//
// One persistent CTA (256 threads) per (sequence, head) at a time.  Thread
// (kb, vb) = (tid / 16, tid % 16) holds the 8x8 tile rows 8 kb.., columns
// 8 vb.. of S and of dS in registers.  Sums over V are warp-shuffle
// transpose-reductions over the 16 lanes of a row group; sums over K go
// through shared memory.  The state at every chunk start is kept in the
// workspace (first, forward pass); then, chunk by chunk from the last, the
// chunk is recomputed forward from its checkpoint (the state before each
// token to a per-CTA scratch, u and d to shared memory) and walked backwards.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int NT = 256;
constexpr int C = kChunk;
constexpr int DK = kHeadK;
constexpr int DV = kHeadV;
constexpr int64_t kTileBytes = (int64_t)DK * DV * 4;     // one state, 64 KiB
constexpr int kMaxCtas = 256;                             // persistent CTAs (scratch slots)

struct BwdArgs {
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
    const float* init;      // [N,H,K,V] or nullptr
    const float* dfinal;    // [N,H,K,V] or nullptr
    float* dq;              // holds dq^ until the norm pass
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    float* dinit;           // or nullptr
    const int32_t* hdr;     // plan header (chunk offsets)
    float4* ckpt;           // (T/64 + N) * H states
    float4* scratch;        // gridDim.x * 64 states
    int32_t* status;
};

__device__ __forceinline__ float ld1(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }

template <typename T>
__device__ __forceinline__ void ld8(const T* p, int64_t i, float (&x)[8])
{
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = ld1(p, i + e);
}

// A state tile in the workspace: float4 q (row 2 q / 2.. of the thread's tile)
// of thread tid at (q * NT + tid): coalesced across the CTA.
__device__ __forceinline__ void tile_store(float4* base, int tid, const float (&s)[64])
{
#pragma unroll
    for (int q = 0; q < 16; ++q)
        base[q * NT + tid] = make_float4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
}
__device__ __forceinline__ void tile_load(const float4* base, int tid, float (&s)[64])
{
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const float4 x = base[q * NT + tid];
        s[4 * q] = x.x; s[4 * q + 1] = x.y; s[4 * q + 2] = x.z; s[4 * q + 3] = x.w;
    }
}

// Sum of x[i] over the 16 lanes of this row group; the lane ends with the sum
// for index 4 h1 + 2 h2 + h3 (h1, h2, h3 = lane bits 3, 2, 1), as does its
// neighbour lane ^ 1.
__device__ __forceinline__ float vsum16(const float (&x)[8], int lane, int& idx)
{
    const int h1 = (lane >> 3) & 1, h2 = (lane >> 2) & 1, h3 = (lane >> 1) & 1;
    float y4[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float keep = h1 ? x[4 + m] : x[m], send = h1 ? x[m] : x[4 + m];
        y4[m] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float y2[2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const float keep = h2 ? y4[2 + m] : y4[m], send = h2 ? y4[m] : y4[2 + m];
        y2[m] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float y1 = (h3 ? y2[1] : y2[0]) + __shfl_xor_sync(0xffffffffu, h3 ? y2[0] : y2[1], 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    idx = 4 * h1 + 2 * h2 + h3;
    return y1;
}

template <typename TIn, typename TO>
__global__ void __launch_bounds__(NT, 1) chunk_bwd_kernel(BwdArgs a)
{
    extern __shared__ float4 dyn_smem[];
    float (*dl_s)[DV] = reinterpret_cast<float (*)[DV]>(dyn_smem);   // d_t of the chunk's tokens
    float (*u_s)[DV] = dl_s + C;                                      // u_t
    __shared__ float red[NT / 32][DV];     // K-reduction partials
    __shared__ float bc[DV];               // broadcast of a per-column result
    __shared__ float rq_s[C], rk_s[C], db_s[C];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kb = tid >> 4, vb = tid & 15;
    const int H = a.H;
    const TIn* gq = static_cast<const TIn*>(a.q);
    const TIn* gk = static_cast<const TIn*>(a.k);
    const TIn* gv = static_cast<const TIn*>(a.v);
    const TO* gdo = static_cast<const TO*>(a.dout);
    float4* scratch = a.scratch + (int64_t)blockIdx.x * C * (kTileBytes / 16);

    // Sum over K of p[j] (this thread's 8 columns): after the call, thread
    // j < DV (the reducer) holds column j's sum in the return value.
    auto ksum = [&](float (&p)[8]) -> float {
#pragma unroll
        for (int j = 0; j < 8; ++j) p[j] += __shfl_xor_sync(0xffffffffu, p[j], 16);
        if (lane < 16) {
#pragma unroll
            for (int j = 0; j < 8; ++j) red[warp][8 * vb + j] = p[j];
        }
        __syncthreads();
        float s = 0.f;
        if (tid < DV) {
#pragma unroll
            for (int w = 0; w < NT / 32; ++w) s += red[w][tid];
        }
        return s;
    };
    // row norms of the chunk's q and k (8 tokens per warp)
    auto chunk_norms = [&](int t0, int L, int h) {
        for (int tl = warp; tl < L; tl += NT / 32) {
            const int64_t base = ((int64_t)(t0 + tl) * H + h) * DK;
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float xq = ld1(gq, base + 4 * lane + e), xk = ld1(gk, base + 4 * lane + e);
                sq += xq * xq;
                sk += xk * xk;
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, m);
                sk += __shfl_xor_sync(0xffffffffu, sk, m);
            }
            if (lane == 0) {
                rq_s[tl] = a.l2norm ? 1.f / sqrtf(sq + 1e-6f) : 1.f;
                rk_s[tl] = a.l2norm ? 1.f / sqrtf(sk + 1e-6f) : 1.f;
                db_s[tl] = 0.f;
            }
        }
        __syncthreads();
    };
    // One forward token: S <- S' + k^ d^T with S' = Diag(a) S.  Stores u and d
    // of the token in u_s / dl_s row `slot` when `keep`.
    auto fwd_token = [&](float (&S)[64], int64_t t, int h, int tl, int slot, bool keep) {
        const int64_t rowk = (t * H + h) * DK + 8 * kb;
        float ga[8], kn[8];
        ld8(a.g, rowk, ga);
        ld8(gk, rowk, kn);
        const float rk = rk_s[tl];
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float ai = expf(ga[i]);
            kn[i] *= rk;
#pragma unroll
            for (int j = 0; j < 8; ++j) S[8 * i + j] *= ai;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc += S[8 * i + j] * kn[i];
            p[j] = acc;
        }
        const float u = ksum(p);
        if (tid < DV) {
            const float d = a.beta[t * H + h] * (ld1(gv, (t * H + h) * DV + tid) - u);
            bc[tid] = d;
            if (keep) {
                u_s[slot][tid] = u;
                dl_s[slot][tid] = d;
            }
        }
        __syncthreads();
        float d8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) d8[j] = bc[8 * vb + j];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) S[8 * i + j] += kn[i] * d8[j];
        __syncthreads();                               // bc and red reused next token
    };

    const int64_t units = (int64_t)a.N * H;
    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int n = (int)(unit / H), h = (int)(unit % H);
        const int bos = a.cu[n], eos = a.cu[n + 1];
        if (bos < 0 || eos < bos || (int64_t)eos > a.T) continue;   // reported by the plan
        const int nch = (eos - bos + C - 1) / C;
        float4* ck = a.ckpt + ((int64_t)a.hdr[kPlanOffsets + n] * H + h) * (kTileBytes / 16);
        const int64_t ck_stride = (int64_t)H * (kTileBytes / 16);

        // ---- forward pass: the state at every chunk start
        float S[64];
        if (a.init != nullptr) {
            const float* s0 = a.init + unit * DK * DV;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) S[8 * i + j] = s0[(8 * kb + i) * DV + 8 * vb + j];
        } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) S[e] = 0.f;
        }
        for (int c = 0; c < nch; ++c) {
            const int t0 = bos + c * C, L = min(C, eos - t0);
            tile_store(ck + c * ck_stride, tid, S);
            chunk_norms(t0, L, h);
            for (int tl = 0; tl < L; ++tl) fwd_token(S, t0 + tl, h, tl, 0, false);
        }

        // ---- backward, chunk by chunk from the last
        float dS[64];
        if (a.dfinal != nullptr) {
            const float* d0 = a.dfinal + unit * DK * DV;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) dS[8 * i + j] = d0[(8 * kb + i) * DV + 8 * vb + j];
        } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) dS[e] = 0.f;
        }
        for (int c = nch - 1; c >= 0; --c) {
            const int t0 = bos + c * C, L = min(C, eos - t0);
            // recompute the chunk: the state before each token, u and d
            tile_load(ck + c * ck_stride, tid, S);
            chunk_norms(t0, L, h);
            for (int tl = 0; tl < L; ++tl) {
                tile_store(scratch + (int64_t)tl * (kTileBytes / 16), tid, S);
                fwd_token(S, t0 + tl, h, tl, tl, true);
            }
            // walk it backwards
            for (int tl = L - 1; tl >= 0; --tl) {
                const int64_t t = t0 + tl;
                const int64_t rowk = (t * H + h) * DK + 8 * kb;
                const int64_t rowv = (t * H + h) * DV + 8 * vb;
                float Sp[64];
                tile_load(scratch + (int64_t)tl * (kTileBytes / 16), tid, Sp);
                float ga[8], kn[8], qn[8], dO[8], d8[8];
                ld8(a.g, rowk, ga);
                ld8(gk, rowk, kn);
                ld8(gq, rowk, qn);
                ld8(gdo, rowv, dO);
                const float rk = rk_s[tl], rq = rq_s[tl], bt = a.beta[t * H + h];
#pragma unroll
                for (int j = 0; j < 8; ++j) d8[j] = dl_s[tl][8 * vb + j];
                float av[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    av[i] = expf(ga[i]);
                    kn[i] *= rk;
                    qn[i] *= rq;
#pragma unroll
                    for (int j = 0; j < 8; ++j) Sp[8 * i + j] *= av[i];
                }
                // o = scale S^T q^:  dS += scale q^ dO^T,  dq^ = scale S dO
                float dqn[8], ddp[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        acc += (Sp[8 * i + j] + kn[i] * d8[j]) * dO[j];
                        dS[8 * i + j] += a.scale * qn[i] * dO[j];
                    }
                    dqn[i] = a.scale * acc;
                }
                // dd = dS^T k^
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc += dS[8 * i + j] * kn[i];
                    ddp[j] = acc;
                }
                const float dd = ksum(ddp);
                if (tid < DV) {
                    const float u = u_s[tl][tid];
                    const float vj = ld1(gv, (t * H + h) * DV + tid);
                    a.dv[(t * H + h) * DV + tid] = bt * dd;
                    bc[tid] = -bt * dd;                        // du
                    float part = dd * (vj - u);
#pragma unroll
                    for (int m = 16; m > 0; m >>= 1) part += __shfl_xor_sync(0xffffffffu, part, m);
                    if (lane == 0) atomicAdd(&db_s[tl], part);
                }
                __syncthreads();
                float du[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) du[j] = bc[8 * vb + j];
                // dk^ = dS d + S' du;  dS' = dS + k^ du^T;  dg = rowsum(dS' o S');  dS = a dS'
                float dkn[8], dgp[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float acc = 0.f, accg = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        acc += dS[8 * i + j] * d8[j] + Sp[8 * i + j] * du[j];
                        const float dsp = dS[8 * i + j] + kn[i] * du[j];
                        accg += dsp * Sp[8 * i + j];
                        dS[8 * i + j] = av[i] * dsp;
                    }
                    dkn[i] = acc;
                    dgp[i] = accg;
                }
                int idx;
                const float sq = vsum16(dqn, lane, idx);
                const float sk = vsum16(dkn, lane, idx);
                const float sg = vsum16(dgp, lane, idx);
                if ((lane & 1) == 0) {
                    const int64_t o = (t * H + h) * DK + 8 * kb + idx;
                    a.dq[o] = sq;
                    a.dk[o] = sk;
                    a.dg[o] = sg;
                }
                __syncthreads();                               // bc reused next token
            }
            for (int tl = tid; tl < L; tl += NT) a.dbeta[(int64_t)(t0 + tl) * H + h] = db_s[tl];
            __syncthreads();
        }
        if (a.dinit != nullptr) {
            float* d0 = a.dinit + unit * DK * DV;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) d0[(8 * kb + i) * DV + 8 * vb + j] = dS[8 * i + j];
        }
    }
}

// dx = (dx^ - x^ (x^ . dx^)) / n with n = sqrt(|x|^2 + eps), in place on dx
// (which holds dx^); one warp per (token, head) row of 128.
template <typename TIn>
__global__ void __launch_bounds__(256) norm_vjp_kernel(const TIn* __restrict__ x,
                                                       float* __restrict__ dx, int64_t rows)
{
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nw) {
        float xv[4], gv[4];
        float ss = 0.f, dot = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            xv[e] = ld1(x, r * DK + 4 * lane + e);
            gv[e] = dx[r * DK + 4 * lane + e];
            ss += xv[e] * xv[e];
            dot += xv[e] * gv[e];
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, m);
            dot += __shfl_xor_sync(0xffffffffu, dot, m);
        }
        const float inv = 1.f / sqrtf(ss + 1e-6f);
        const float proj = dot * inv * inv;                 // (x^ . dx^) / n
#pragma unroll
        for (int e = 0; e < 4; ++e) dx[r * DK + 4 * lane + e] = (gv[e] - xv[e] * proj) * inv;
    }
}

template <typename TIn, typename TO>
cudaError_t launch_typed(const BwdArgs& a, int grid, cudaStream_t stream)
{
    constexpr int smem = 2 * C * DV * 4;
    cudaError_t e = cudaFuncSetAttribute(chunk_bwd_kernel<TIn, TO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_bwd_kernel<TIn, TO><<<grid, NT, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess || !a.l2norm || a.T == 0) return e;
    const int64_t rows = a.T * a.H;
    const int sms = device_sm_count();
    int64_t blocks = std::min<int64_t>((rows + 7) / 8, (int64_t)(sms > 0 ? sms : 152) * 8);
    norm_vjp_kernel<TIn><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const TIn*>(a.q),
                                                                a.dq, rows);
    norm_vjp_kernel<TIn><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const TIn*>(a.k),
                                                                a.dk, rows);
    return cudaGetLastError();
}

}  // namespace

int64_t bwd_workspace_bytes(int32_t N, int64_t T, int32_t H)
{
    const int64_t ctas = std::min<int64_t>((int64_t)N * H, kMaxCtas);
    return chunk_plan_header_bytes(N) + split_chunk_bound(N, T) * H * kTileBytes +
           ctas * C * kTileBytes;
}

cudaError_t launch_chunk_bwd(const BwdLaunch& L, cudaStream_t stream)
{
    const int64_t units = (int64_t)L.N * L.H;
    const int sms = device_sm_count();
    const int grid = (int)std::min<int64_t>(units, std::min<int64_t>(kMaxCtas, sms > 0 ? sms : 152));
    int32_t* hdr = static_cast<int32_t*>(L.workspace);
    unsigned char* ws = static_cast<unsigned char*>(L.workspace) + chunk_plan_header_bytes(L.N);
    BwdArgs a;
    a.q = L.q; a.k = L.k; a.v = L.v; a.qkv_bf16 = L.qkv_bf16; a.g = L.g; a.beta = L.beta;
    a.cu = L.cu; a.N = L.N; a.T = L.T; a.H = L.H; a.scale = L.scale; a.l2norm = L.l2norm;
    a.dout = L.dout; a.dout_bf16 = L.dout_bf16; a.init = L.init; a.dfinal = L.dfinal;
    a.dq = L.dq; a.dk = L.dk; a.dv = L.dv; a.dg = L.dg; a.dbeta = L.dbeta; a.dinit = L.dinit;
    a.hdr = hdr;
    a.ckpt = reinterpret_cast<float4*>(ws);
    a.scratch = reinterpret_cast<float4*>(ws + split_chunk_bound(L.N, L.T) * L.H * kTileBytes);
    a.status = L.status;
    cudaError_t e = launch_chunk_plan(L.cu, L.N, L.T, hdr, L.status, stream);
    if (e != cudaSuccess || units == 0) return e;
    if (L.qkv_bf16)
        return L.dout_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(a, grid, stream)
                           : launch_typed<__nv_bfloat16, float>(a, grid, stream);
    return L.dout_bf16 ? launch_typed<float, __nv_bfloat16>(a, grid, stream)
                       : launch_typed<float, float>(a, grid, stream);
}

}  // namespace kda
