// Tensor-core chunked KDA forward (tcgen05, TMEM accumulators), sm_103a.
//
// One CTA (256 threads) per (sequence, head); chunks of 64 tokens in order.
// The state is carried transposed, S^T (V x K = 128 x 128): its FP32 master
// lives in registers (thread (v, half) holds S^T[v][64 half .. 64 half + 63])
// and a BF16 copy in shared memory is the A operand of the next chunk's MMAs.
// Every MMA has M = 128 (the V or K dimension) so D occupies all 128 TMEM lanes.
//
// Per chunk (the chunk solve of "Add opt-in FP32 KDA chunk computation",
// sections Problem and Change, in its WY form):
//   prep (CUDA cores)  q^, k^ (L2 norm), a = e^g, A_kk, A_qk (overflow-safe
//                      factors, as in the FP32 kernel), T = (I + A_kk)^-1
//                      by 16x16 blocks, X = beta k^ o e^G, Q' = q^ o e^G,
//                      K'' = k^ o e^{G_last - G}, d = e^{G_last}
//   MMA (TF32)         W^T = X^T T^T,  U^T = (beta V)^T T^T
//   MMA (BF16)         [W S]^T = S^T W^T,  [Q' S]^T = S^T Q'^T
//   epilogue           Delta^T = U^T - [W S]^T
//   MMA (TF32)         O^T += Delta^T Aqk^T,  P^T = Delta^T K''
//   epilogue           out = scale O;  S^T <- S^T Diag(d) + P^T
//
// Operand precision: the state-side products (W S, Q' S) take BF16 operands;
// every product inside the chunk (T, Delta, A_qk, K'') takes TF32 operands,
// because BF16 rounding there alone costs about 1.6e-3 of output rel-L2 (FP64
// emulation of this algorithm), which with a BF16 output would exceed the
// 3e-3 budget.  Accumulation is FP32 in TMEM throughout.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = kChunk;     // 64
constexpr int DK = kHeadK;    // 128
constexpr int DV = kHeadV;    // 128
constexpr int NT = 256;
constexpr int LDW = 132;      // fp32 work-row stride (floats)
constexpr int LDA = C + 1;
constexpr int SB = 16;
constexpr int NB = C / SB;
constexpr uint32_t kWaitIters = 1u << 22;   // polls before a wait gives up

// Shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t WORK_BYTES = C * LDW * 4;              // 33792 = 33 KiB
constexpr uint32_t OFF_ST = 0;                            // S^T bf16 [128][128]   32 KiB
constexpr uint32_t OFF_QW = OFF_ST + 32768;               // q work -> Q' bf16 | T tf32
constexpr uint32_t OFF_KW = OFF_QW + WORK_BYTES;          // k work -> X^T tf32 -> W bf16 (MN)
constexpr uint32_t OFF_AW = OFF_KW + WORK_BYTES;          // e^g -> k^ o bwd -> K''^T tf32
constexpr uint32_t OFF_VW = OFF_AW + WORK_BYTES;          // v work -> (beta V)^T tf32 -> Delta^T
constexpr uint32_t OFF_AQK = OFF_VW + WORK_BYTES;         // A_qk tf32 [64][64]    16 KiB
constexpr uint32_t OFF_AKK = OFF_AQK + 16384;             // A_kk fp32 [64][65]
constexpr uint32_t OFF_TF = OFF_AKK + C * LDA * 4;        // T fp32 [64][65]
constexpr uint32_t OFF_BLK = OFF_TF + C * LDA * 4;        // blk fp32 [4][128]
constexpr uint32_t OFF_DEC = OFF_BLK + NB * DK * 4;       // d fp32 [128]
constexpr uint32_t OFF_BETA = OFF_DEC + DK * 4;           // beta fp32 [64]
constexpr uint32_t OFF_BAR = OFF_BETA + C * 4;            // 3 mbarriers + TMEM slot + flag
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;         // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_QW % 1024 == 0 && OFF_KW % 1024 == 0 && OFF_AW % 1024 == 0 &&
              OFF_VW % 1024 == 0 && OFF_AQK % 1024 == 0, "SW128 tiles need 1024-B alignment");
constexpr uint32_t OFF_QP = OFF_QW;                        // Q' bf16 [64][128], 16 KiB
constexpr uint32_t OFF_TT = OFF_QW + 16384;                // T tf32 [64][64], 16 KiB

// TMEM columns.
constexpr uint32_t TM_WS = 0, TM_O = 64, TM_P = 128, TM_W = 256, TM_U = 320, TM_COLS = 512;

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// 8 consecutive input elements -> float.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8])
{
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8])
{
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p + 4));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NT, 1) chunk_tc_kernel(ChunkArgs args)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    unsigned char* sm = smem_raw + pad;
    const uint32_t sb = raw_s + pad;                      // shared-window address of sm

    float (*Qw)[LDW] = reinterpret_cast<float (*)[LDW]>(sm + OFF_QW);
    float (*Kw)[LDW] = reinterpret_cast<float (*)[LDW]>(sm + OFF_KW);
    float (*Aw)[LDW] = reinterpret_cast<float (*)[LDW]>(sm + OFF_AW);
    float (*Vw)[LDW] = reinterpret_cast<float (*)[LDW]>(sm + OFF_VW);
    float (*akk)[LDA] = reinterpret_cast<float (*)[LDA]>(sm + OFF_AKK);
    float (*Tf)[LDA] = reinterpret_cast<float (*)[LDA]>(sm + OFF_TF);
    float (*blk)[DK] = reinterpret_cast<float (*)[DK]>(sm + OFF_BLK);
    float* dec = reinterpret_cast<float*>(sm + OFF_DEC);
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);   // [0] prep, [1] S1, [2] S3
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 32);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane;                     // TMEM lane = V (or K) index
    const int n = blockIdx.x / args.H, h = blockIdx.x % args.H;
    const int H = args.H;

    const int bos = args.cu_seqlens[n], eos = args.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || (int64_t)eos > args.T) {
        if (tid == 0) report_status(args.status, KDA_ERR_DEVICE_ARG);
        return;
    }
    const TIn* __restrict__ gq = static_cast<const TIn*>(args.q);
    const TIn* __restrict__ gk = static_cast<const TIn*>(args.k);
    const TIn* __restrict__ gv = static_cast<const TIn*>(args.v);
    TOut* __restrict__ out = static_cast<TOut*>(args.out);

    // ---- setup: zero S^T, TMEM allocation, barriers
    for (int e = tid; e < 32768 / 16; e += NT)
        reinterpret_cast<uint4*>(sm + OFF_ST)[e] = make_uint4(0, 0, 0, 0);
    if (warp == 0) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 3; ++b) mbar_init(&bar[b], 1);
        fence_mbar_init();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tlane = tmem + ((uint32_t)(32 * quad) << 16);

    float S[64];                                           // S^T[row][64 half + c]
#pragma unroll
    for (int c = 0; c < 64; ++c) S[c] = 0.f;
    bool failed = false;
    int last_bar = -1;                                     // last barrier committed to
    uint32_t phase = 0;

    for (int t0 = bos; t0 < eos && !failed; t0 += C, phase ^= 1u) {
        const int L = min(C, eos - t0);

        // ---- P1: load the chunk (rows >= L: zero, decay factor 1); zero A_qk
        for (int e = tid; e < C * (DK / 8); e += NT) {
            const int r = e / (DK / 8), c8 = (e % (DK / 8)) * 8;
            float xq[8], xk[8], xv[8], xa[8];
            if (r < L) {
                const int64_t off = ((int64_t)(t0 + r) * H + h) * DK + c8;
                load8(gq + off, xq);
                load8(gk + off, xk);
                load8(gv + ((int64_t)(t0 + r) * H + h) * DV + c8, xv);
                const float4 g0 = __ldg(reinterpret_cast<const float4*>(args.g + off));
                const float4 g1 = __ldg(reinterpret_cast<const float4*>(args.g + off + 4));
                xa[0] = expf(g0.x); xa[1] = expf(g0.y); xa[2] = expf(g0.z); xa[3] = expf(g0.w);
                xa[4] = expf(g1.x); xa[5] = expf(g1.y); xa[6] = expf(g1.z); xa[7] = expf(g1.w);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) { xq[i] = 0.f; xk[i] = 0.f; xv[i] = 0.f; xa[i] = 1.f; }
            }
#pragma unroll
            for (int i = 0; i < 8; i += 4) {
                *reinterpret_cast<float4*>(&Qw[r][c8 + i]) = make_float4(xq[i], xq[i + 1], xq[i + 2], xq[i + 3]);
                *reinterpret_cast<float4*>(&Kw[r][c8 + i]) = make_float4(xk[i], xk[i + 1], xk[i + 2], xk[i + 3]);
                *reinterpret_cast<float4*>(&Vw[r][c8 + i]) = make_float4(xv[i], xv[i + 1], xv[i + 2], xv[i + 3]);
                *reinterpret_cast<float4*>(&Aw[r][c8 + i]) = make_float4(xa[i], xa[i + 1], xa[i + 2], xa[i + 3]);
            }
        }
        if (tid < C) sbeta[tid] = tid < L ? args.beta[(int64_t)(t0 + tid) * H + h] : 0.f;
        for (int e = tid; e < 16384 / 16; e += NT)
            reinterpret_cast<uint4*>(sm + OFF_AQK)[e] = make_uint4(0, 0, 0, 0);
        __syncthreads();

        // ---- P2: L2 normalisation (warp per row)
        if (args.l2norm) {
            for (int r = warp; r < C; r += NT / 32) {
                float sq = 0.f, sk = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float x = Qw[r][lane + 32 * m], y = Kw[r][lane + 32 * m];
                    sq += x * x;
                    sk += y * y;
                }
                sq = warp_sum(sq);
                sk = warp_sum(sk);
                const float iq = 1.f / sqrtf(sq + 1e-6f), ik = 1.f / sqrtf(sk + 1e-6f);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    Qw[r][lane + 32 * m] *= iq;
                    Kw[r][lane + 32 * m] *= ik;
                }
            }
            __syncthreads();
        }

        // ---- P3: pairs inside one 16-token block (running products of a_t)
        for (int j = warp; j < C; j += NT / 32) {
            const int bend = (j / SB) * SB + SB;
            float kp[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) kp[m] = Kw[j][lane + 32 * m];
            for (int i = j; i < bend; ++i) {
                float skk = 0.f, sqk = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = lane + 32 * m;
                    if (i > j) kp[m] *= Aw[i][c];
                    skk += Kw[i][c] * kp[m];
                    sqk += Qw[i][c] * kp[m];
                }
                skk = warp_sum(skk);
                sqk = warp_sum(sqk);
                if (lane == 0) {
                    akk[i][j] = (i > j) ? sbeta[i] * skk : 0.f;
                    *reinterpret_cast<float*>(sm + OFF_AQK + sw128_tile(64, i, j * 4)) = sqk;
                }
            }
        }
        __syncthreads();

        // ---- P4: per channel, products inside each block (fwd / bwd / totals)
        if (tid < DK) {
            const int c = tid;
            float tot = 1.f;
            for (int I = 0; I < NB; ++I) {
                float av[SB], kk[SB];
                float p = 1.f;
#pragma unroll
                for (int u = 0; u < SB; ++u) {
                    const int r = I * SB + u;
                    av[u] = Aw[r][c];
                    kk[u] = Kw[r][c];
                    p *= av[u];
                    Qw[r][c] *= p;
                    Kw[r][c] = kk[u] * p;
                }
                blk[I][c] = p;
                tot *= p;
                float pb = 1.f;
#pragma unroll
                for (int u = SB - 1; u >= 0; --u) {
                    Aw[I * SB + u][c] = kk[u] * pb;
                    pb *= av[u];
                }
            }
            dec[c] = tot;
        }
        __syncthreads();

        // ---- P5: pairs in different blocks
        for (int e = tid; e < 6 * SB * SB; e += NT) {
            const int pi = e / (SB * SB);
            const int I = pi == 0 ? 1 : (pi < 3 ? 2 : 3);
            const int J = pi == 0 ? 0 : (pi < 3 ? pi - 1 : pi - 3);
            const int i = I * SB + (e % (SB * SB)) / SB;
            const int j = J * SB + e % SB;
            float skk = 0.f, sqk = 0.f;
            for (int c = 0; c < DK; ++c) {
                float mid = 1.f;
                for (int M = J + 1; M < I; ++M) mid *= blk[M][c];
                const float kb = Aw[j][c] * mid;
                skk += Kw[i][c] * kb;
                sqk += Qw[i][c] * kb;
            }
            akk[i][j] = sbeta[i] * skk;
            *reinterpret_cast<float*>(sm + OFF_AQK + sw128_tile(64, i, j * 4)) = sqk;
        }
        __syncthreads();

        // ---- P6: T = (I + A_kk)^-1 by 16x16 blocks
        if (warp < NB && lane < SB) {          // diagonal blocks, one warp each
            const int b = warp * SB, m = lane;
            float tcol[SB];
#pragma unroll
            for (int i = 0; i < SB; ++i) {
                float acc = (i == m) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) acc -= akk[b + i][b + j] * tcol[j];
                tcol[i] = (i < m) ? 0.f : acc;
            }
#pragma unroll
            for (int i = 0; i < SB; ++i) Tf[b + i][b + m] = tcol[i];
        }
        __syncthreads();
        for (int d = 1; d < NB; ++d) {
            // Y_IJ = sum_{M=J}^{I-1} A_IM T_MJ, kept in the unused block (J, I) of Tf
            for (int e = tid; e < (NB - d) * SB * SB; e += NT) {
                const int J = e / (SB * SB), I = J + d;
                const int r = (e % (SB * SB)) / SB, cc = e % SB;
                float acc = 0.f;
                for (int M = J; M < I; ++M)
                    for (int k = 0; k < SB; ++k)
                        acc += akk[I * SB + r][M * SB + k] * Tf[M * SB + k][J * SB + cc];
                Tf[J * SB + r][I * SB + cc] = acc;
            }
            __syncthreads();
            // T_IJ = -T_II Y_IJ
            for (int e = tid; e < (NB - d) * SB * SB; e += NT) {
                const int J = e / (SB * SB), I = J + d;
                const int r = (e % (SB * SB)) / SB, cc = e % SB;
                float acc = 0.f;
                for (int k = 0; k <= r; ++k) acc += Tf[I * SB + r][I * SB + k] * Tf[J * SB + k][I * SB + cc];
                Tf[I * SB + r][J * SB + cc] = -acc;
            }
            __syncthreads();
        }

        // ---- P7: MMA operands.  Read everything needed into registers first.
        {
            // X^T[c][j] = beta_j k^_jc e^{G_jc}, K''^T[c][j] = k^_jc e^{G_last,c - G_jc},
            // Q'[i][c] = q^_ic e^{G_ic}, (beta V)^T[v][j]; T tf32.
            float xv[32], kv[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int e = tid + u * NT;
                const int j = e / DK, c = e % DK, J = j / SB;
                float pre = 1.f, post = 1.f;
                for (int M = 0; M < J; ++M) pre *= blk[M][c];
                for (int M = J + 1; M < NB; ++M) post *= blk[M][c];
                xv[u] = sbeta[j] * Kw[j][c] * pre;
                kv[u] = Aw[j][c] * post;
                Qw[j][c] *= pre;                          // Q' in place (fp32)
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int e = tid + u * NT;
                const int j = e / DK, c = e % DK;
                *reinterpret_cast<float*>(sm + OFF_KW + sw128_tile(128, c, j * 4)) = xv[u];
                *reinterpret_cast<float*>(sm + OFF_AW + sw128_tile(128, c, j * 4)) = kv[u];
            }
            float vv[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int e = tid + u * NT;
                const int j = e / DV, m = e % DV;
                vv[u] = sbeta[j] * Vw[j][m];
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int e = tid + u * NT;
                const int j = e / DV, m = e % DV;
                *reinterpret_cast<float*>(sm + OFF_VW + sw128_tile(128, m, j * 4)) = vv[u];
            }
        }
        __syncthreads();
        // Q' bf16 K-major [64 i][128 c] (Q' fp32 still in Qw rows; written to the
        // first 16 KiB of the same region after a register round trip).
        {
            uint32_t qp[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int e = tid + u * NT;
                const int i = e / 64, c2 = (e % 64) * 2;
                qp[u] = pack_bf16(Qw[i][c2], Qw[i][c2 + 1]);
            }
            float tt[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int e = tid + u * NT;
                const int i = e / 64, j = e % 64;
                tt[u] = (j <= i) ? Tf[i][j] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int e = tid + u * NT;
                const int i = e / 64, c2 = (e % 64) * 2;
                *reinterpret_cast<uint32_t*>(sm + OFF_QP + sw128_tile(64, i, c2 * 2)) = qp[u];
                const int j = e % 64;
                *reinterpret_cast<float*>(sm + OFF_TT + sw128_tile(64, i, j * 4)) = tt[u];
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- P8: W^T = X^T T^T, U^T = (beta V)^T T^T  (TF32)
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t id = idesc(kFmtTF32, 128, 64);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_tf32(tmem + TM_W, desc_kmajor(sb + OFF_KW, 128, s), desc_kmajor(sb + OFF_TT, 64, s), id, s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_tf32(tmem + TM_U, desc_kmajor(sb + OFF_VW, 128, s), desc_kmajor(sb + OFF_TT, 64, s), id, s > 0);
            commit(&bar[0]);
        }
        last_bar = 0;
        {
            const bool ok = mbar_wait(&bar[0], phase, kWaitIters);
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        fence_after_sync();
        // W bf16, MN-major [c][i] (row c = TMEM lane, 32 tokens per half)
        {
            float w[32];
            tmem_ld32(tlane + TM_W + 32 * half, w);
            unsigned char* dst = sm + OFF_KW;
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                uint4 pk;
                pk.x = pack_bf16(w[8 * q8 + 0], w[8 * q8 + 1]);
                pk.y = pack_bf16(w[8 * q8 + 2], w[8 * q8 + 3]);
                pk.z = pack_bf16(w[8 * q8 + 4], w[8 * q8 + 5]);
                pk.w = pack_bf16(w[8 * q8 + 6], w[8 * q8 + 7]);
                *reinterpret_cast<uint4*>(dst + sw128(row, (32 * half + 8 * q8) * 2)) = pk;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- S1: [W S]^T = S^T W^T, [Q' S]^T = S^T Q'^T  (BF16)
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t idw = idesc(kFmtBF16, 128, 64, false, true);
            constexpr uint32_t idq = idesc(kFmtBF16, 128, 64);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tmem + TM_WS, desc_kmajor(sb + OFF_ST, 128, s), desc_mnmajor64(sb + OFF_KW, s), idw, s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tmem + TM_O, desc_kmajor(sb + OFF_ST, 128, s), desc_kmajor(sb + OFF_QP, 64, s), idq, s > 0);
            commit(&bar[1]);
        }
        last_bar = 1;
        {
            const bool ok = mbar_wait(&bar[1], phase, kWaitIters);
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        fence_after_sync();
        // Delta^T[v][i] = U^T[v][i] - [W S]^T[v][i], TF32 operand K-major [v][i]
        {
            float ws[32], uu[32];
            tmem_ld32(tlane + TM_WS + 32 * half, ws);
            tmem_ld32(tlane + TM_U + 32 * half, uu);
            unsigned char* dst = sm + OFF_VW;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 dv = make_float4(uu[4 * q4] - ws[4 * q4], uu[4 * q4 + 1] - ws[4 * q4 + 1],
                                              uu[4 * q4 + 2] - ws[4 * q4 + 2], uu[4 * q4 + 3] - ws[4 * q4 + 3]);
                *reinterpret_cast<float4*>(dst + sw128_tile(128, row, (32 * half + 4 * q4) * 4)) = dv;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- S3: O^T += Delta^T Aqk^T, P^T = Delta^T K''  (TF32)
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t ido = idesc(kFmtTF32, 128, 64);
            constexpr uint32_t idp = idesc(kFmtTF32, 128, 128);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_tf32(tmem + TM_O, desc_kmajor(sb + OFF_VW, 128, s), desc_kmajor(sb + OFF_AQK, 64, s), ido, 1);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_tf32(tmem + TM_P, desc_kmajor(sb + OFF_VW, 128, s), desc_kmajor(sb + OFF_AW, 128, s), idp, s > 0);
            commit(&bar[2]);
        }
        last_bar = 2;
        {
            const bool ok = mbar_wait(&bar[2], phase, kWaitIters);
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        fence_after_sync();
        // out = scale * O;  S^T <- S^T Diag(d) + P^T;  BF16 copy of S^T for the next chunk
        {
            float o[32];
            tmem_ld32(tlane + TM_O + 32 * half, o);
            const int v = row;
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                const int i = 32 * half + u;
                if (i < L) store_out(out + ((int64_t)(t0 + i) * H + h) * DV + v, args.scale * o[u]);
            }
            float p[32];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                tmem_ld32(tlane + TM_P + 64 * half + 32 * part, p);
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int c = 64 * half + 32 * part + u;
                    S[32 * part + u] = S[32 * part + u] * dec[c] + p[u];
                }
            }
            unsigned char* dst = sm + OFF_ST;
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                uint4 pk;
                pk.x = pack_bf16(S[8 * q8 + 0], S[8 * q8 + 1]);
                pk.y = pack_bf16(S[8 * q8 + 2], S[8 * q8 + 3]);
                pk.z = pack_bf16(S[8 * q8 + 4], S[8 * q8 + 5]);
                pk.w = pack_bf16(S[8 * q8 + 6], S[8 * q8 + 7]);
                *reinterpret_cast<uint4*>(dst + sw128_tile(128, row, (64 * half + 8 * q8) * 2)) = pk;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
    }

    if (failed) {
        if (tid == 0) report_status(args.status, KDA_ERR_TIMEOUT);
        // let the MMAs still in flight finish before the TMEM is released
        if (last_bar >= 0) mbar_wait(&bar[last_bar], phase, kWaitIters);
    } else if (args.final_state != nullptr) {
        float* fs = args.final_state + ((int64_t)n * H + h) * DK * DV;
#pragma unroll
        for (int u = 0; u < 64; ++u) fs[(int64_t)(64 * half + u) * DV + row] = S[u];
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

template <typename TIn, typename TOut>
cudaError_t launch_typed(const ChunkArgs& a, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel<TIn, TOut>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.N * a.H;
    if (units > INT32_MAX) return cudaErrorInvalidConfiguration;
    chunk_tc_kernel<TIn, TOut><<<(unsigned)units, NT, SMEM_BYTES, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t stream)
{
    if (a.qkv_bf16)
        return a.out_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(a, stream)
                          : launch_typed<__nv_bfloat16, float>(a, stream);
    return a.out_bf16 ? launch_typed<float, __nv_bfloat16>(a, stream)
                      : launch_typed<float, float>(a, stream);
}

}  // namespace kda
