// State-free steps of one 64-token chunk on the tensor-core path, shared by
// the single-pass kernel (kda_chunk_tc.cu) and the chunk-preparation kernel
// of the two-phase path (kda_chunk_split.cu).  Every function here assumes a
// CTA of 256 threads and is called by all of them.
//
// With G the in-chunk prefix of the log-decay g and a_t = e^{g_t}, one chunk
// needs ("Add opt-in FP32 KDA chunk computation", sections Problem and Change):
//   A_kk[i][j] = beta_i sum_c k^_ic k^_jc e^{G_ic - G_jc}   (j < i)
//   A_qk[i][j] =        sum_c q^_ic k^_jc e^{G_ic - G_jc}   (j <= i)
//   T' = (I + A_kk)^-1 diag(beta)
// The pair sums are formed without overflow as a binary tree of "straddle"
// levels (kda_chunk_tc.cu describes the factorisation); each level's operands
// are FP16 rows of 128 channels in 128-byte-swizzled tiles.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace chunk_ops {

using tc::sw128;

constexpr int C = kChunk;     // 64
constexpr int DK = kHeadK;    // 128
constexpr int NT = 256;       // threads per CTA
constexpr int LDA = C + 4;    // fp32 row stride of A_kk and T: 16-byte aligned rows
constexpr int SB = 16;        // diagonal block of the inverse
constexpr int NB = C / SB;

// Staging keeps 16-bit activations: BF16 inputs as they are, FP32 inputs
// rounded to FP16 (the MMA operands are FP16 anyway).
template <typename TIn> struct Stage;
template <> struct Stage<__nv_bfloat16> {
    __device__ static float to_f32(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }
};
template <> struct Stage<float> {
    __device__ static float to_f32(uint16_t x) { return __half2float(__ushort_as_half(x)); }
};

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack_h8(const float* v)
{
    uint4 pk;
    pk.x = pack_h2(v[0], v[1]);
    pk.y = pack_h2(v[2], v[3]);
    pk.z = pack_h2(v[4], v[5]);
    pk.w = pack_h2(v[6], v[7]);
    return pk;
}

// 8 FP16 values at MN indices m .. m+7 (m % 8 == 0) of K row `row` of a
// 128-byte-swizzled tile whose 64-element MN groups are `gbytes` apart.
// The tile may live in shared or in global memory.
__device__ __forceinline__ void st8(unsigned char* tile, uint32_t gbytes, int row, int m,
                                    const float* v)
{
    *reinterpret_cast<uint4*>(tile + (m >> 6) * gbytes + sw128(row, (m & 63) * 2)) = pack_h8(v);
}

// One 16-byte piece of a chunk row, global -> staging (rows >= L are zero).
template <typename TIn> struct Loader;
template <> struct Loader<__nv_bfloat16> {
    static constexpr int kPieces = DK / 8;          // 16-byte pieces per 128-element row
    __device__ static uint4 load(const __nv_bfloat16* row, int piece)
    {
        return __ldg(reinterpret_cast<const uint4*>(row) + piece);
    }
    __device__ static void store(unsigned char* stage, int r, int piece, uint4 x)
    {
        *reinterpret_cast<uint4*>(stage + r * 256 + piece * 16) = x;
    }
};
template <> struct Loader<float> {
    static constexpr int kPieces = DK / 4;
    __device__ static uint4 load(const float* row, int piece)
    {
        return __ldg(reinterpret_cast<const uint4*>(row) + piece);
    }
    __device__ static void store(unsigned char* stage, int r, int piece, uint4 x)
    {
        uint2 hx;
        hx.x = pack_h2(__uint_as_float(x.x), __uint_as_float(x.y));
        hx.y = pack_h2(__uint_as_float(x.z), __uint_as_float(x.w));
        *reinterpret_cast<uint2*>(stage + r * 256 + piece * 8) = hx;
    }
};

// Row norms and q^ . k^ of the staged chunk (4 threads per row, 32 channels
// each): rq = 1/|q_t|, rk = 1/|k_t| (1 without normalisation), dqk = q^_t . k^_t.
template <typename TIn>
__device__ __forceinline__ void chunk_norms(const unsigned char* sq, const unsigned char* sk,
                                            float* rq, float* rk, float* dqk, bool l2norm,
                                            int tid)
{
    using ST = Stage<TIn>;
    const int r = tid >> 2, p4 = tid & 3;
    float s2q = 0.f, s2k = 0.f, sqk = 0.f;
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
        const int piece = p4 + 4 * ((i4 + r) & 3);   // 16-byte piece of the row
        const uint4 uq = *reinterpret_cast<const uint4*>(sq + r * 256 + piece * 16);
        const uint4 uk = *reinterpret_cast<const uint4*>(sk + r * 256 + piece * 16);
        const uint32_t wq[4] = {uq.x, uq.y, uq.z, uq.w}, wk[4] = {uk.x, uk.y, uk.z, uk.w};
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) {
            const float q0 = ST::to_f32((uint16_t)(wq[w2] & 0xffffu));
            const float q1 = ST::to_f32((uint16_t)(wq[w2] >> 16));
            const float k0 = ST::to_f32((uint16_t)(wk[w2] & 0xffffu));
            const float k1 = ST::to_f32((uint16_t)(wk[w2] >> 16));
            s2q += q0 * q0 + q1 * q1;
            s2k += k0 * k0 + k1 * k1;
            sqk += q0 * k0 + q1 * k1;
        }
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        s2q += __shfl_xor_sync(0xffffffffu, s2q, o);
        s2k += __shfl_xor_sync(0xffffffffu, s2k, o);
        sqk += __shfl_xor_sync(0xffffffffu, sqk, o);
    }
    if (p4 == 0) {
        const float iq = l2norm ? 1.f / sqrtf(s2q + 1e-6f) : 1.f;
        const float ik = l2norm ? 1.f / sqrtf(s2k + 1e-6f) : 1.f;
        rq[r] = iq;
        rk[r] = ik;
        dqk[r] = iq * ik * sqk;
    }
}

// The per-channel rows of channel c over this thread's 32 tokens (32 hh + u):
//   X'^T = k^ o e^G and Q' = q^ o e^G (prefix decay within the chunk, `before`
//   = decay of the tokens before this thread's half), K''^T = k^ o e^{G_last - G}
//   (suffix decay, `after` = decay of the tokens after this thread's half).
// Each goes to row c of a 128-byte-swizzled [128 c][64 j] FP16 tile, in
// shared or global memory.
__device__ __forceinline__ void channel_rows(unsigned char* xt, unsigned char* qp,
                                             unsigned char* kt, int c, int hh, float before,
                                             float after, const float (&a)[32],
                                             const float (&kh)[32], const float (&qh)[32])
{
    float p = before;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float x1[8], x2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            p *= a[8 * q + e];
            x1[e] = kh[8 * q + e] * p;
            x2[e] = qh[8 * q + e] * p;
        }
        st8(xt, 0, c, 32 * hh + 8 * q, x1);
        st8(qp, 0, c, 32 * hh + 8 * q, x2);
    }
    p = after;
#pragma unroll
    for (int q = 3; q >= 0; --q) {
        float x1[8];
#pragma unroll
        for (int e = 7; e >= 0; --e) {
            x1[e] = kh[8 * q + e] * p;
            p *= a[8 * q + e];
        }
        st8(kt, 0, c, 32 * hh + 8 * q, x1);
    }
}

// Writes one level's left (upper-half) and right (lower-half) operand rows for
// channel c over this thread's 32 tokens (a, kh, qh hold tokens 32 hh + u).
// Level S <= 16: both halves of every 2S-block lie in this thread's 32 tokens,
// and its 16 upper (and 16 lower) tokens have level indices 16 hh .. 16 hh + 15.
// Values are formed and stored 8 at a time to keep few registers live.
template <int S>
__device__ __forceinline__ void level_operands(unsigned char* buf, int c, int hh, int mo, int no,
                                               const float (&a)[32], const float (&kh)[32],
                                               const float (&qh)[32])
{
    unsigned char* A = buf;
    unsigned char* B = buf + 32768;
    float p = 1.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {                    // upper: forward from the midpoint
        float lk[8], lq[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int li = 8 * q + e, x = li % S, up = 2 * S * (li / S) + S;
            p = (x == 0) ? a[up] : p * a[up + x];
            lk[e] = kh[up + x] * p;
            lq[e] = qh[up + x] * p;
        }
        st8(A, 16384, c, mo + 16 * hh + 8 * q, lk);
        st8(A, 16384, c, mo + 32 + 16 * hh + 8 * q, lq);
    }
#pragma unroll
    for (int q = 1; q >= 0; --q) {                   // lower: backward to the midpoint
        float rr[8];
#pragma unroll
        for (int e = 7; e >= 0; --e) {
            const int li = 8 * q + e, x = li % S, lo = 2 * S * (li / S);
            if (x == S - 1) {
                rr[e] = kh[lo + x];
                p = a[lo + x];
            } else {
                rr[e] = kh[lo + x] * p;
                p *= a[lo + x];
            }
        }
        st8(B, 16384, c, no + 16 * hh + 8 * q, rr);
    }
}

// Level 32: the upper half (tokens 32..63) is thread hh = 1, the lower hh = 0.
__device__ __forceinline__ void level32_operands(unsigned char* buf, int c, int hh,
                                                 const float (&a)[32], const float (&kh)[32],
                                                 const float (&qh)[32])
{
    unsigned char* A = buf;
    unsigned char* B = buf + 32768;
    if (hh == 1) {
        float p = 1.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float v1[8], v2[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int x = 8 * q + e;
                p = (x == 0) ? a[0] : p * a[x];
                v1[e] = kh[x] * p;
                v2[e] = qh[x] * p;
            }
            st8(A, 16384, c, 8 * q, v1);
            st8(A, 16384, c, 32 + 8 * q, v2);
        }
    } else {
        float p = 1.f;
#pragma unroll
        for (int q = 3; q >= 0; --q) {
            float v1[8];
#pragma unroll
            for (int e = 7; e >= 0; --e) {
                const int x = 8 * q + e;
                if (x == 31) {
                    v1[e] = kh[x];
                    p = a[x];
                } else {
                    v1[e] = kh[x] * p;
                    p *= a[x];
                }
            }
            st8(B, 16384, c, 8 * q, v1);
        }
    }
}

// Pair sums of level S for the 32 TMEM lanes of this warp: lane u is upper
// token index u of the level; r holds columns [16 hf, 16 hf + 16) of the
// level's 32 right (lower-half) tokens.  The valid columns of a lane are one
// contiguous run of j (the lower half of its block), written with vector
// stores: k rows to A_kk (fp32, row stride LDA, times beta_i), q rows to the
// A_qk tile (fp16, 128-byte swizzled [64 i][64 j]).  Only entries j < i.
template <int S>
__device__ __forceinline__ void extract_level(unsigned char* aqk, float* akk, const float* beta,
                                              const float* r, int u, int hf, bool qrows)
{
    constexpr int W = S < 16 ? S : 16;                    // valid columns per lane
    constexpr int NCASE = S < 16 ? 16 / S : 1;            // blocks per 16-column window
    const int bi = u / S;                                 // block of this lane's token
    const int i = bi * 2 * S + S + (u % S);
    int j0;
    bool valid;
    if (S == 32) { j0 = 16 * hf; valid = true; }
    else if (S == 16) { j0 = 32 * bi; valid = (bi == hf); }
    else { j0 = 2 * S * bi; valid = ((bi * S) >> 4) == hf; }
    if (!valid) return;
    float v[W];
    const int cs = (S < 16) ? (bi & (NCASE - 1)) : 0;     // which block of the window
#pragma unroll
    for (int x = 0; x < W; ++x) {
        float t = r[x];
#pragma unroll
        for (int c = 1; c < NCASE; ++c) t = (cs == c) ? r[c * S + x] : t;
        v[x] = t;
    }
    if (qrows) {
        unsigned char* dst = aqk + sw128(i, j0 * 2);
        if constexpr (W >= 8) {
#pragma unroll
            for (int q = 0; q < W / 8; ++q)
                *reinterpret_cast<uint4*>(aqk + sw128(i, (j0 + 8 * q) * 2)) = pack_h8(v + 8 * q);
        } else if constexpr (W == 4) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]));
        } else if constexpr (W == 2) {
            *reinterpret_cast<uint32_t*>(dst) = pack_h2(v[0], v[1]);
        } else {
            *reinterpret_cast<__half*>(dst) = __float2half_rn(v[0]);
        }
    } else {
        const float beta_i = beta[i];
        float* dst = akk + i * LDA + j0;
        if constexpr (W >= 4) {
#pragma unroll
            for (int q = 0; q < W / 4; ++q)
                reinterpret_cast<float4*>(dst)[q] =
                    make_float4(beta_i * v[4 * q], beta_i * v[4 * q + 1], beta_i * v[4 * q + 2],
                                beta_i * v[4 * q + 3]);
        } else if constexpr (W == 2) {
            *reinterpret_cast<float2*>(dst) = make_float2(beta_i * v[0], beta_i * v[1]);
        } else {
            *dst = beta_i * v[0];
        }
    }
}

// Zeroes the strictly upper part of the A_qk tile (disjoint from the entries
// the extraction writes).
__device__ __forceinline__ void aqk_zero_upper(unsigned char* aqk, int tid)
{
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int e = tid + u * NT;                       // 512 pieces of 8 columns
        const int i = e >> 3, p8 = e & 7;
        unsigned char* dst = aqk + sw128(i, p8 * 16);
        if (8 * p8 > i) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        } else if (8 * p8 + 7 > i) {
#pragma unroll
            for (int x = 0; x < 8; ++x)
                if (8 * p8 + x > i) reinterpret_cast<__half*>(dst)[x] = __float2half_rn(0.f);
        }
    }
}

// All six levels from the three pair-sum accumulators (TMEM columns
// [tm_a, tm_a + 192)) of this thread's lanes, plus the A_qk diagonal.
__device__ __forceinline__ void extract_pairs(unsigned char* aqk, float* akk, const float* beta,
                                              const float* dqk, uint32_t tlane, uint32_t tm_a,
                                              int tid, int warp, int lane)
{
    const int quad = warp & 3, half = warp >> 2;
    const bool second = quad >= 2, qrows = (quad & 1) != 0;
    const uint32_t tb = tlane + tm_a + (second ? 32 : 0) + 16 * half;
    float r[48];
    tc::tmem_ld16x3(tb, tb + 64, tb + 128, r);
    if (second) {
        extract_level<16>(aqk, akk, beta, r, lane, half, qrows);
        extract_level<4>(aqk, akk, beta, r + 16, lane, half, qrows);
        extract_level<1>(aqk, akk, beta, r + 32, lane, half, qrows);
    } else {
        extract_level<32>(aqk, akk, beta, r, lane, half, qrows);
        extract_level<8>(aqk, akk, beta, r + 16, lane, half, qrows);
        extract_level<2>(aqk, akk, beta, r + 32, lane, half, qrows);
    }
    if (tid < C) *reinterpret_cast<__half*>(aqk + sw128(tid, tid * 2)) = __float2half_rn(dqk[tid]);
}

// T = (I + A_kk)^-1 by blocks: 16x16 diagonal blocks by forward substitution,
// then the 32- and 64-row merges T_BA = -T_B A_BA T_A (Y scratch kept in the
// unused upper blocks of T); finally T' = T diag(beta) as an FP16 K-major
// [64 i][64 j] tile.  Entry: A_kk complete and visible (after a CTA barrier).
// Exit: the T' tile written by this thread (the caller fences and syncs).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float f4(const float4& v, int e)
{
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// Rows of A_kk and T are read 4 columns at a time (16-byte loads along k);
// every accumulation keeps its k order.  chunk_inverse_f32 leaves T in Tf
// (FP32, unit diagonal; its upper blocks hold scratch and must be read as 0)
// and ends with a CTA barrier.
__device__ __forceinline__ void chunk_inverse_f32(float (*akk)[LDA], float (*Tf)[LDA], int tid,
                                                  int warp, int lane)
{
    if (warp < NB && lane < SB) {
        const int b = warp * SB, m = lane;
        float tcol[SB];
#pragma unroll
        for (int i = 0; i < SB; ++i) {
            float acc = (i == m) ? 1.f : 0.f;
#pragma unroll
            for (int q = 0; q < (i + 3) / 4; ++q) {
                const float4 a4 = ld4(&akk[b + i][b + 4 * q]);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * q + e < i) acc -= f4(a4, e) * tcol[4 * q + e];
            }
            tcol[i] = (i < m) ? 0.f : acc;
        }
#pragma unroll
        for (int i = 0; i < SB; ++i) Tf[b + i][b + m] = tcol[i];
    }
    __syncthreads();
    {
        // 32-row merges for blocks (1,0) and (3,2): Y = A_{I,I-1} T_{I-1,I-1}
        // (one 2x1 micro-tile per thread; Y kept in the unused block (I-1, I))
        const int blk = tid >> 7, I = 1 + 2 * blk, J = I - 1;
        const int r2 = ((tid >> 4) & 7) * 2, cc = tid & 15;
        float y0 = 0.f, y1 = 0.f;
#pragma unroll
        for (int q = 0; q < SB / 4; ++q) {
            const float4 a0 = ld4(&akk[I * SB + r2][J * SB + 4 * q]);
            const float4 a1 = ld4(&akk[I * SB + r2 + 1][J * SB + 4 * q]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float t = Tf[J * SB + 4 * q + e][J * SB + cc];
                y0 += f4(a0, e) * t;
                y1 += f4(a1, e) * t;
            }
        }
        Tf[J * SB + r2][I * SB + cc] = y0;
        Tf[J * SB + r2 + 1][I * SB + cc] = y1;
        __syncthreads();
        float t0 = 0.f, t1 = 0.f;
#pragma unroll
        for (int q = 0; q < SB / 4; ++q) {
            const float4 b0 = ld4(&Tf[I * SB + r2][I * SB + 4 * q]);
            const float4 b1 = ld4(&Tf[I * SB + r2 + 1][I * SB + 4 * q]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float y = Tf[J * SB + 4 * q + e][I * SB + cc];
                t0 += f4(b0, e) * y;
                t1 += f4(b1, e) * y;
            }
        }
        Tf[I * SB + r2][J * SB + cc] = -t0;
        Tf[I * SB + r2 + 1][J * SB + cc] = -t1;
    }
    __syncthreads();
    {
        // 64-row merge: Y = A[32:64, 0:32] T[0:32, 0:32] (kept in Tf[0:32, 32:64]),
        // then T[32:64, 0:32] = -T[32:64, 32:64] Y; one 2x2 micro-tile per thread
        const int r2 = (tid >> 4) * 2, c2 = (tid & 15) * 2;
        const int k0 = c2 < SB ? 0 : SB;            // T[0:32,0:32] is zero above its blocks
        float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
#pragma unroll 2
        for (int k = k0; k < 32; k += 4) {
            const float4 a0 = ld4(&akk[32 + r2][k]), a1 = ld4(&akk[32 + r2 + 1][k]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 t = *reinterpret_cast<const float2*>(&Tf[k + e][c2]);
                y00 += f4(a0, e) * t.x; y01 += f4(a0, e) * t.y;
                y10 += f4(a1, e) * t.x; y11 += f4(a1, e) * t.y;
            }
        }
        *reinterpret_cast<float2*>(&Tf[r2][32 + c2]) = make_float2(y00, y01);
        *reinterpret_cast<float2*>(&Tf[r2 + 1][32 + c2]) = make_float2(y10, y11);
        __syncthreads();
        const int k1 = r2 < SB ? SB : 32;            // T[32:64,32:64] likewise
        float t00 = 0.f, t01 = 0.f, t10 = 0.f, t11 = 0.f;
#pragma unroll 2
        for (int k = 0; k < k1; k += 4) {
            const float4 b0 = ld4(&Tf[32 + r2][32 + k]), b1 = ld4(&Tf[32 + r2 + 1][32 + k]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 y = *reinterpret_cast<const float2*>(&Tf[k + e][32 + c2]);
                t00 += f4(b0, e) * y.x; t01 += f4(b0, e) * y.y;
                t10 += f4(b1, e) * y.x; t11 += f4(b1, e) * y.y;
            }
        }
        *reinterpret_cast<float2*>(&Tf[32 + r2][c2]) = make_float2(-t00, -t01);
        *reinterpret_cast<float2*>(&Tf[32 + r2 + 1][c2]) = make_float2(-t10, -t11);
    }
    __syncthreads();
}

// kBetaInTp: beta lies inside the T' tile, so each thread reads its beta_j
// before the inverse's last barrier (once T' is being written it is gone).
template <bool kBetaInTp = false>
__device__ __forceinline__ void chunk_inverse(float (*akk)[LDA], float (*Tf)[LDA],
                                              const float* sbeta, unsigned char* tp, int tid,
                                              int warp, int lane)
{
    float4 bq[2][2];
    auto read_beta = [&] {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int j0 = ((tid + u * NT) % 8) * 8;
            bq[u][0] = ld4(sbeta + j0);
            bq[u][1] = ld4(sbeta + j0 + 4);
        }
    };
    if constexpr (kBetaInTp) read_beta();
    chunk_inverse_f32(akk, Tf, tid, warp, lane);
    if constexpr (!kBetaInTp) read_beta();
    // T'[i][j] = T[i][j] beta_j (j <= i), row i, 8 columns per store
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int e = tid + u * NT;                  // 512 pieces of 8
        const int i = e / 8, j0 = (e % 8) * 8;
        const float4 ta = ld4(&Tf[i][j0]), tb = ld4(&Tf[i][j0 + 4]);
        const float4 ba = bq[u][0], bb = bq[u][1];
        float v8[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const float tv = x < 4 ? f4(ta, x) : f4(tb, x - 4);
            const float bv = x < 4 ? f4(ba, x) : f4(bb, x - 4);
            v8[x] = (j0 + x <= i) ? tv * bv : 0.f;
        }
        st8(tp, 0, i, j0, v8);
    }
}

}  // namespace chunk_ops
}  // namespace kda
