// FP32-exact chunked KDA forward on CUDA cores (IEEE FP32 throughout).
//
// One CTA per (sequence, head, 64-wide slice of V).  Chunks of 64 tokens
// start at the sequence start and are processed in order; the state slice
// S[:, v0:v0+64] (128 x 64 FP32) stays in shared memory for the whole
// sequence.  Per chunk, with G_i the in-chunk inclusive prefix of g
// (per channel) and D = Diag(exp G_last):
//
//   A_ij   = beta_i sum_c k_ic k_jc e^{G_ic - G_jc}          (j < i)
//   Aqk_ij =        sum_c q_ic k_jc e^{G_ic - G_jc}          (j <= i)
//   (I + A) [W | U] = [diag(beta) (K o e^G) | diag(beta) V]  (forward substitution)
//   Delta = U - W S
//   O     = scale [ (Q o e^G) S + Aqk Delta ]
//   S    <- D S + (K o e^{G_last - G})^T Delta
//
// This is the chunk solve of the pages' chunked KDA ("Add opt-in FP32 KDA
// chunk computation", sections Problem and Change: chunk solve and state
// intermediates kept in FP32, Q/K L2-normalised inside the op).
//
// Overflow-safe decay factors.  e^{G_i} e^{-G_j} overflows FP32 long before
// e^{G_i - G_j} <= 1 does (in-chunk decays reach e^{-1000}), and G_i - G_j
// taken from two large prefixes loses digits.  So no factor is ever formed
// from a difference of prefixes: every factor is a running product of the
// per-token decays a_t = e^{g_t} <= 1 over the tokens it spans.  The chunk is
// split into four 16-token blocks; for i in block I and j in block J < I,
//   e^{G_i - G_j} = bwd_j * mid_{IJ} * fwd_i,
//   fwd_i = prod_{t = start(I)}^{i} a_t,   bwd_j = prod_{t = j+1}^{end(J)} a_t,
//   mid_{IJ} = product of the totals of the blocks strictly between J and I,
// every factor <= 1.  Pairs inside one block use running products directly.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = kChunk;        // 64
constexpr int DK = kHeadK;       // 128
constexpr int BV = 64;           // V slice per CTA
constexpr int NVS = kHeadV / BV; // slices per head
constexpr int NT = 256;
constexpr int LDK = DK + 4;
constexpr int LDV = BV + 4;
constexpr int LDA = C + 1;
constexpr int SB = 16;           // sub-block
constexpr int NB = C / SB;       // 4 sub-blocks

struct Smem {
    float q[C][LDK];     // q^ -> q^ o fwd -> Q' = q^ o e^G
    float k[C][LDK];     // k^ -> k^ o fwd -> X = beta k^ o e^G -> W
    float a[C][LDK];     // e^g -> k^ o bwd -> K'' = k^ o e^{G_last - G}
    float v[C][LDV];     // v slice -> beta v -> U
    float akk[C][LDA];
    float aqk[C][LDA];
    float s[DK][LDV];    // state slice
    float dlt[C][LDV];   // Delta
    float blk[NB][DK];   // per sub-block total decay
    float dec[DK];       // e^{G_last}
    float beta[C];
};

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename TIn, typename TOut, int kGate>
__global__ void __launch_bounds__(NT, 1) chunk_fp32_kernel(ChunkArgs args)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t unit = blockIdx.x;                 // ((n * H) + h) * NVS + vs
    const int vs = (int)(unit % NVS);
    const int h = (int)((unit / NVS) % args.H);
    const int n = (int)(unit / ((int64_t)NVS * args.H));
    const int H = args.H;
    const int v0 = vs * BV;

    const int bos = args.cu_seqlens[n], eos = args.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || (int64_t)eos > args.T) {
        if (tid == 0) report_status(args.status, KDA_ERR_DEVICE_ARG);
        return;
    }
    const TIn* __restrict__ q = static_cast<const TIn*>(args.q);
    const TIn* __restrict__ k = static_cast<const TIn*>(args.k);
    const TIn* __restrict__ v = static_cast<const TIn*>(args.v);
    const float* __restrict__ g = args.g;
    TOut* __restrict__ out = static_cast<TOut*>(args.out);

    if (args.initial_state != nullptr) {
        const float* s0 = args.initial_state + ((int64_t)n * H + h) * DK * kHeadV;
        for (int i = tid; i < DK * BV; i += NT)
            sm.s[i / BV][i % BV] = s0[(int64_t)(i / BV) * kHeadV + v0 + i % BV];
    } else {
        for (int i = tid; i < DK * BV; i += NT) sm.s[i / BV][i % BV] = 0.f;
    }
    constexpr bool kGated = kGate != kGateG;
    using TG = typename GateSrc<kGate>::T;                 // element of g or f
    const TG* __restrict__ graw =
        kGated ? static_cast<const TG*>(args.f) : reinterpret_cast<const TG*>(g);
    const float lamneg = kGated ? -expf(args.A_log[h]) : 0.f;

    for (int t0 = bos; t0 < eos; t0 += C) {
        const int L = min(C, eos - t0);
        __syncthreads();

        // ---- 1. load the chunk; rows past the sequence end are zero (decay 1)
        for (int i = tid; i < C * DK; i += NT) {
            const int r = i / DK, c = i % DK;
            float qv = 0.f, kv = 0.f, av = 1.f;
            if (r < L) {
                const int64_t off = ((int64_t)(t0 + r) * H + h) * DK + c;
                qv = load_as_float(q + off);
                kv = load_as_float(k + off);
                const float gin = load_as_float(graw + off);
                av = expf(kGated ? gate_decay(gin, args.dt_bias[(int64_t)h * DK + c], lamneg) : gin);
            }
            sm.q[r][c] = qv;
            sm.k[r][c] = kv;
            sm.a[r][c] = av;
        }
        for (int i = tid; i < C * BV; i += NT) {
            const int r = i / BV, m = i % BV;
            float vv = 0.f;
            if (r < L) vv = load_as_float(v + ((int64_t)(t0 + r) * H + h) * kHeadV + v0 + m);
            sm.v[r][m] = vv;
        }
        if (tid < C) {
            float bt = 0.f;
            if (tid < L) {
                const int64_t i = (int64_t)(t0 + tid) * H + h;
                if (kGated)
                    bt = gate_sigmoid(args.b_bf16
                                          ? __bfloat162float(static_cast<const __nv_bfloat16*>(args.b)[i])
                                          : static_cast<const float*>(args.b)[i]);
                else
                    bt = args.beta[i];
            }
            sm.beta[tid] = bt;
        }
        __syncthreads();

        // ---- 2. L2 normalisation of q and k rows (one warp per row)
        if (args.l2norm) {
            for (int r = warp; r < C; r += NT / 32) {
                float sq = 0.f, sk = 0.f;
                for (int c = lane; c < DK; c += 32) {
                    const float x = sm.q[r][c], y = sm.k[r][c];
                    sq += x * x;
                    sk += y * y;
                }
                sq = warp_sum(sq);
                sk = warp_sum(sk);
                const float iq = 1.f / sqrtf(sq + 1e-6f), ik = 1.f / sqrtf(sk + 1e-6f);
                for (int c = lane; c < DK; c += 32) {
                    sm.q[r][c] *= iq;
                    sm.k[r][c] *= ik;
                }
            }
            __syncthreads();
        }

        // ---- 3. pairs inside one 16-token block: running products of a_t
        for (int j = warp; j < C; j += NT / 32) {
            const int bend = (j / SB) * SB + SB;
            float kp[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) kp[m] = sm.k[j][lane + 32 * m];
            for (int i = j; i < bend; ++i) {
                float skk = 0.f, sqk = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = lane + 32 * m;
                    if (i > j) kp[m] *= sm.a[i][c];
                    skk += sm.k[i][c] * kp[m];
                    sqk += sm.q[i][c] * kp[m];
                }
                skk = warp_sum(skk);
                sqk = warp_sum(sqk);
                if (lane == 0) {
                    sm.akk[i][j] = (i > j) ? sm.beta[i] * skk : 0.f;
                    sm.aqk[i][j] = sqk;
                }
            }
        }
        __syncthreads();

        // ---- 4. per channel: fwd/bwd products inside each block
        if (tid < DK) {
            const int c = tid;
            float tot = 1.f;
            for (int I = 0; I < NB; ++I) {
                float av[SB], kk[SB];
                float p = 1.f;
#pragma unroll
                for (int u = 0; u < SB; ++u) {
                    const int r = I * SB + u;
                    av[u] = sm.a[r][c];
                    kk[u] = sm.k[r][c];
                    p *= av[u];
                    sm.q[r][c] *= p;               // q^ o fwd
                    sm.k[r][c] = kk[u] * p;        // k^ o fwd
                }
                sm.blk[I][c] = p;
                tot *= p;
                float pb = 1.f;
#pragma unroll
                for (int u = SB - 1; u >= 0; --u) {
                    sm.a[I * SB + u][c] = kk[u] * pb;   // k^ o bwd
                    pb *= av[u];
                }
            }
            sm.dec[c] = tot;
        }
        __syncthreads();

        // ---- 5. pairs in different blocks: (k^ o fwd)_i . mid . (k^ o bwd)_j
        for (int e = tid; e < 6 * SB * SB; e += NT) {
            const int pi = e / (SB * SB);
            // (I, J) for pi = 0..5: (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
            const int I = pi == 0 ? 1 : (pi < 3 ? 2 : 3);
            const int J = pi == 0 ? 0 : (pi < 3 ? pi - 1 : pi - 3);
            const int i = I * SB + (e % (SB * SB)) / SB;
            const int j = J * SB + e % SB;
            float skk = 0.f, sqk = 0.f;
            for (int c = 0; c < DK; ++c) {
                float mid = 1.f;
                for (int M = J + 1; M < I; ++M) mid *= sm.blk[M][c];
                const float kb = sm.a[j][c] * mid;
                skk += sm.k[i][c] * kb;
                sqk += sm.q[i][c] * kb;
            }
            sm.akk[i][j] = sm.beta[i] * skk;
            sm.aqk[i][j] = sqk;
        }
        __syncthreads();

        // ---- 6. X = beta k^ o e^G, Q' = q^ o e^G, K'' = k^ o e^{G_last - G}, beta v
        for (int i = tid; i < C * DK; i += NT) {
            const int r = i / DK, c = i % DK, I = r / SB;
            float pre = 1.f, post = 1.f;
            for (int M = 0; M < I; ++M) pre *= sm.blk[M][c];
            for (int M = I + 1; M < NB; ++M) post *= sm.blk[M][c];
            sm.k[r][c] *= sm.beta[r] * pre;
            sm.q[r][c] *= pre;
            sm.a[r][c] *= post;
        }
        for (int i = tid; i < C * BV; i += NT) sm.v[i / BV][i % BV] *= sm.beta[i / BV];
        __syncthreads();

        // ---- 7. (I + A)[W | U] = [X | beta V], forward substitution over rows
        for (int i = 1; i < L; ++i) {
            for (int col = tid; col < DK + BV; col += NT) {
                float acc = 0.f;
                if (col < DK) {
                    for (int j = 0; j < i; ++j) acc += sm.akk[i][j] * sm.k[j][col];
                    sm.k[i][col] -= acc;
                } else {
                    const int m = col - DK;
                    for (int j = 0; j < i; ++j) acc += sm.akk[i][j] * sm.v[j][m];
                    sm.v[i][m] -= acc;
                }
            }
            __syncthreads();
        }

        // ---- 8. Delta = U - W S
        for (int e = tid; e < C * BV; e += NT) {
            const int i = e / BV, m = e % BV;
            float acc = 0.f;
            if (i < L)
                for (int c = 0; c < DK; ++c) acc += sm.k[i][c] * sm.s[c][m];
            sm.dlt[i][m] = (i < L) ? sm.v[i][m] - acc : 0.f;
        }
        __syncthreads();

        // ---- 9. O = scale [Q' S + Aqk Delta]; new state into registers
        for (int e = tid; e < L * BV; e += NT) {
            const int i = e / BV, m = e % BV;
            float acc = 0.f, acc2 = 0.f;
            for (int c = 0; c < DK; ++c) acc += sm.q[i][c] * sm.s[c][m];
            for (int j = 0; j <= i; ++j) acc2 += sm.aqk[i][j] * sm.dlt[j][m];
            store_out(out + ((int64_t)(t0 + i) * H + h) * kHeadV + v0 + m,
                      args.scale * (acc + acc2));
        }
        float snew[DK * BV / NT];
#pragma unroll 4
        for (int u = 0; u < DK * BV / NT; ++u) {
            const int e = tid + u * NT;
            const int c = e / BV, m = e % BV;
            float acc = sm.dec[c] * sm.s[c][m];
            for (int j = 0; j < L; ++j) acc += sm.a[j][c] * sm.dlt[j][m];
            snew[u] = acc;
        }
        __syncthreads();
#pragma unroll 4
        for (int u = 0; u < DK * BV / NT; ++u) {
            const int e = tid + u * NT;
            sm.s[e / BV][e % BV] = snew[u];
        }
    }
    __syncthreads();
    if (args.final_state != nullptr) {
        float* fs = args.final_state + ((int64_t)n * H + h) * DK * kHeadV;
        for (int e = tid; e < DK * BV; e += NT) {
            const int c = e / BV, m = e % BV;
            fs[(int64_t)c * kHeadV + v0 + m] = sm.s[c][m];
        }
    }
}

template <typename TIn, typename TOut, int kGate>
cudaError_t launch_typed(const ChunkArgs& a, cudaStream_t stream)
{
    const size_t smem = sizeof(Smem);
    cudaError_t e = cudaFuncSetAttribute(chunk_fp32_kernel<TIn, TOut, kGate>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.N * a.H * NVS;
    if (units > INT32_MAX) return cudaErrorInvalidConfiguration;
    chunk_fp32_kernel<TIn, TOut, kGate><<<(unsigned)units, NT, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int kGate>
cudaError_t launch_gated(const ChunkArgs& a, cudaStream_t stream)
{
    if (a.qkv_bf16)
        return a.out_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16, kGate>(a, stream)
                          : launch_typed<__nv_bfloat16, float, kGate>(a, stream);
    return a.out_bf16 ? launch_typed<float, __nv_bfloat16, kGate>(a, stream)
                      : launch_typed<float, float, kGate>(a, stream);
}

}  // namespace

cudaError_t launch_chunk_fp32(const ChunkArgs& a, cudaStream_t stream)
{
    switch (gate_in(a)) {
        case kGateF32: return launch_gated<kGateF32>(a, stream);
        case kGateBF16: return launch_gated<kGateBF16>(a, stream);
        default: return launch_gated<kGateG>(a, stream);
    }
}

}  // namespace kda
