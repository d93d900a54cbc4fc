// FP32-exact chunked KDA forward in two phases.
//
// The same split as the tensor-core two-phase path ("Add opt-in FP32 KDA chunk
// computation", sections Problem and Change: the chunk solve and the carried
// state, kept in FP32 here):
//   prepare (every (chunk, head) at once, one CTA each, IEEE FP32 on CUDA
//   cores):
//     A_kk, A_qk (pair sums with decay factors built from 4- and 16-token
//     sub-blocks, each a product of factors <= 1, so that nothing overflows),
//     T = (I + A_kk)^-1 (16x16 blocks and their merges), W = T X with
//     X = beta k^ o e^G, U = T (beta v), Q' = q^ o e^G,
//     K'' = k^ o e^{G_last - G}, d = e^{G_last}   ->  one record
//   scan (one CTA per (sequence, head, half of V), chunks in order, tcgen05):
//     Delta = U - W S,  O = scale [Q' S + A_qk Delta],  S <- Diag(d) S + K''^T Delta
// The scan's products run on the tensor cores with each FP32 operand x held
// as a pair of FP16 values, x ~ (hi + lo) / s: hi = fp16(x s) and
// lo = fp16(x s - hi) carry about 22 significant bits, and
// x y ~ (hi_x hi_y + hi_x lo_y + lo_x hi_y) / (s_x s_y), three MMAs with FP32
// accumulation, the dropped lo_x lo_y term below 2^-22 of the product.  The
// scales s are powers of two (exact): per row of W (whose magnitude follows
// T), per chunk for the state and for Delta (they follow v and beta, so a
// fixed scale would either overflow FP16 or leave small states in its
// subnormals), and 1 for Q', K'' and A_qk (|x| <= 1: unit q^, k^ and decays
// <= 1).  The state itself, U, d, Delta = U - W S and the state update are
// FP32 on CUDA cores.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_chunk_ops.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = kChunk;        // 64
constexpr int DK = kHeadK;       // 128
constexpr int DV = kHeadV;       // 128
constexpr int NT = 256;
constexpr int SB = 16;           // block of the decay factorisation
constexpr int NB = C / SB;
constexpr int S4 = 4;            // sub-block inside a block
constexpr int LDK = DK + 4;      // FP32 rows of 128 (16-byte aligned, shifted banks)
constexpr int LDT = chunk_ops::LDA;   // 68: A_kk and T for the blocked inverse
constexpr int LDQ = C + 4;       // A_qk

// Record of one unit (bytes).  FP16 pairs (hi, lo) are two tiles of the
// same 128-byte-swizzled layout, lo 32 KiB (W, Q'), 16 KiB (K'') or 8 KiB
// (A_qk) after hi.  The scan brings the early part in before [W; Q'] S and
// the late part before K''^T Delta.
constexpr uint32_t R_WQ = 0;           // [W; Q'] K-major [128 rows][128 c]: rows 0..63 W s_i, 64..127 Q'
constexpr uint32_t R_WQ_LO = 32768;
constexpr uint32_t R_WINV = 65536;     // 1 / s_i of W row i, FP32 [64]
constexpr uint32_t R_U = 65792;        // U FP32 [2 halves of V][64 i][64 v], 16-byte piece p of row i at p ^ (i & 7)
constexpr uint32_t R_LATE = R_U + 32768;
constexpr uint32_t L_KT = 0;           // K''^T MN-major [64 i][128 c] (two 64-channel groups of 8 KiB)
constexpr uint32_t L_KT_LO = 16384;
constexpr uint32_t L_AQK = 32768;      // A_qk K-major [64 i][64 j] (zero above the diagonal)
constexpr uint32_t L_AQK_LO = 40960;
constexpr uint32_t L_DEC = 49152;      // d FP32 [128]
constexpr uint32_t R_LATE_BYTES = L_DEC + 512;
constexpr uint32_t R_BYTES = R_LATE + R_LATE_BYTES;
constexpr uint32_t R_UHALF = 16384;
static_assert(R_BYTES % 16 == 0 && R_LATE % 16 == 0 && R_U % 16 == 0, "bulk copy sizes");

// x s as an FP16 pair: hi = fp16(x s), lo = fp16(x s - hi), eight values at
// MN (or K) indices m .. m + 7 of row `row` of a swizzled tile pair (lo at
// hi + lo_off, 64-element groups `gbytes` apart), in shared or global memory.
__device__ __forceinline__ void st8_pair(unsigned char* tile, uint32_t lo_off, uint32_t gbytes,
                                         int row, int m, const float* x, float s)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float y0 = x[2 * e] * s, y1 = x[2 * e + 1] * s;
        const __half2 hh = __floats2half2_rn(y0, y1);
        const float2 hf = __half22float2(hh);
        const __half2 ll = __floats2half2_rn(y0 - hf.x, y1 - hf.y);
        h[e] = *reinterpret_cast<const uint32_t*>(&hh);
        l[e] = *reinterpret_cast<const uint32_t*>(&ll);
    }
    const uint32_t o = (m >> 6) * gbytes + tc::sw128(row, (m & 63) * 2);
    *reinterpret_cast<uint4*>(tile + o) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(tile + lo_off + o) = make_uint4(l[0], l[1], l[2], l[3]);
}

// The power of two s = 2^(14 - e) for a maximum magnitude mx < 2^e, and 1/s:
// every |x| <= mx then has |x s| < 2^14, inside FP16's range with room for
// the rounding of hi.  The exponent is kept within +-100 (mx of zero, or
// beyond FP32's range).
__device__ __forceinline__ void pow2_scale(float mx, float& s, float& inv)
{
    const int e = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 126;
    const int k = max(-100, min(100, 14 - e));
    s = __uint_as_float((uint32_t)(127 + k) << 23);
    inv = __uint_as_float((uint32_t)(127 - k) << 23);
}

struct PrepSmem {
    float q[C][LDK];       // q^ -> Qf4 -> Qf16 (then Q' goes to the record)
    float k[C][LDK];       // k^ -> Kf4 -> Kf16 -> X
    float a[C][LDK];       // e^g -> Kb4 -> Kb16 (then K'' goes to the record)
    float v[C][LDK];       // v -> beta v
    float akk[C][LDT];     // A_kk (beta-scaled, strictly lower)
    float tf[C][LDT];      // T = (I + A_kk)^-1
    float aqk[C][LDQ];
    float t4[C / S4][DK];  // decay over each 4-token sub-block
    float blk[NB][DK];     // decay over each 16-token block
    // the decay over the sub-blocks between two others of a block, by block:
    // [I][0] = 1, [I][1] = t4 of sub-block 1, [I][2] = of 2, [I][3] = of 1 and 2
    float mid4[NB][4][DK];
    float mid16[4][DK];    // likewise over the blocks between two others
    float pre16[NB][DK];   // the decay over the blocks before block I
    float post16[NB][DK];  // over the blocks after it
    float beta[C];
};

__device__ __forceinline__ float4 ld4s(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4s(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float f4at(const float4& v, int e)
{
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}
__device__ __forceinline__ float4 mul4(float4 a, float4 b)
{
    return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}
__device__ __forceinline__ float4 scale4(float4 a, float s)
{
    return make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
}
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc)
{
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

// Eight consecutive elements of a row, raw (16 bytes of BF16 or 32 of FP32).
template <typename T> struct Raw8;
template <> struct Raw8<float> {
    float4 lo, hi;
    __device__ __forceinline__ void load(const float* p)
    {
        lo = *reinterpret_cast<const float4*>(p);
        hi = *reinterpret_cast<const float4*>(p + 4);
    }
    __device__ __forceinline__ void zero() { lo = hi = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ void get(float (&x)[8]) const
    {
        x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
        x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
    }
};
template <> struct Raw8<__nv_bfloat16> {
    uint4 w;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) { w = *reinterpret_cast<const uint4*>(p); }
    __device__ __forceinline__ void zero() { w = make_uint4(0u, 0u, 0u, 0u); }
    __device__ __forceinline__ void get(float (&x)[8]) const
    {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {        // a BF16 is the top half of an FP32
            x[2 * i] = __uint_as_float(u[i] << 16);
            x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
        }
    }
};

// Reduce-scatter of N partial sums over the G lanes (a power of two, aligned
// in the warp) that hold them: afterwards v[0 .. N/G) of lane l are the totals
// of entries (l mod G) * N/G .. + N/G.  Every lane of the warp takes part.
template <int N, int O>
struct ReduceScatter {
    static __device__ __forceinline__ void run(float* v, int lane)
    {
        constexpr int h = N / 2;
        const bool up = (lane & O) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h];
            const float keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
        }
        ReduceScatter<h, O / 2>::run(v, lane);
    }
};
template <int N>
struct ReduceScatter<N, 0> {
    static __device__ __forceinline__ void run(float*, int) {}
};

// ---------------------------------------------------------------- prepare
// Pair sums over a chunk, A[i][j] = sum_c x_i[c] k_j[c] e^{G_i[c] - G_j[c]}
// (j <= i), with every decay factor a product of e^g over a run of tokens
// (each <= 1, so nothing overflows and an underflow only hides a term that is
// below FP32's range anyway):
//   i, j in one 4-token sub-block: running products from j;
//   i, j in different sub-blocks of one 16-token block: (x_i o fwd4_i) .
//     (k_j o bwd4_j o mid4), fwd4 the products from i's sub-block start to i,
//     bwd4 from after j to its sub-block end, mid4 the sub-blocks in between;
//   i, j in different 16-token blocks: the same with 16-token blocks.
template <typename TIn, int kGate>
__global__ void __launch_bounds__(NT, 1) fp32_prep_kernel(ChunkArgs args,
                                                          const int32_t* __restrict__ hdr,
                                                          unsigned char* __restrict__ records)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    PrepSmem& sm = *reinterpret_cast<PrepSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = args.H;
    const int32_t* off = hdr + kPlanOffsets;
    const int64_t unit = blockIdx.x;
    const int32_t gc = (int32_t)(unit / H);
    const int h = (int)(unit % H);
    if (gc >= off[args.N]) return;                        // past the chunks of the offsets
    int lo = 0, hi = args.N - 1;                           // last n with off[n] <= gc
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= gc) lo = mid;
        else hi = mid - 1;
    }
    const int bos = args.cu_seqlens[lo], eos = args.cu_seqlens[lo + 1];
    const int t0 = bos + (gc - off[lo]) * C;
    const int L = min(C, eos - t0);
    unsigned char* recb = records + unit * (int64_t)R_BYTES;

    const TIn* __restrict__ q = static_cast<const TIn*>(args.q);
    const TIn* __restrict__ k = static_cast<const TIn*>(args.k);
    const TIn* __restrict__ v = static_cast<const TIn*>(args.v);
    constexpr bool kGated = kGate != kGateG;
    using TG = typename GateSrc<kGate>::T;
    const TG* __restrict__ graw =
        kGated ? static_cast<const TG*>(args.f) : reinterpret_cast<const TG*>(args.g);

    // ---- 1. the chunk: q^, k^ (row L2 norms over the 16 lanes that hold a
    // row), e^g, v; rows past the sequence end are zero with decay 1
    {
        const int c0 = (tid & 15) * 8;
        float dtb[8];
        float lamneg = 0.f;
        if constexpr (kGated) {
            lamneg = -expf(args.A_log[h]);
            const float4 d0 = *reinterpret_cast<const float4*>(args.dt_bias + (int64_t)h * DK + c0);
            const float4 d1 = *reinterpret_cast<const float4*>(args.dt_bias + (int64_t)h * DK + c0 + 4);
            dtb[0] = d0.x; dtb[1] = d0.y; dtb[2] = d0.z; dtb[3] = d0.w;
            dtb[4] = d1.x; dtb[5] = d1.y; dtb[6] = d1.z; dtb[7] = d1.w;
        }
        Raw8<TIn> rq[4], rk[4], rv[4];
        Raw8<TG> rg[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int r = (tid >> 4) + 16 * m;
            if (r < L) {
                const int64_t o = ((int64_t)(t0 + r) * H + h) * DK + c0;
                rq[m].load(q + o);
                rk[m].load(k + o);
                rv[m].load(v + o);
                rg[m].load(graw + o);
            } else {
                rq[m].zero(); rk[m].zero(); rv[m].zero(); rg[m].zero();
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int r = (tid >> 4) + 16 * m;
            float xq[8], xk[8], xv[8], xg[8];
            rq[m].get(xq); rk[m].get(xk); rv[m].get(xv); rg[m].get(xg);
            if (args.l2norm) {
                float sq = 0.f, sk = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    sq = fmaf(xq[i], xq[i], sq);
                    sk = fmaf(xk[i], xk[i], sk);
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) {
                    sq += __shfl_xor_sync(0xffffffffu, sq, o);
                    sk += __shfl_xor_sync(0xffffffffu, sk, o);
                }
                const float iq = 1.f / sqrtf(sq + 1e-6f), ik = 1.f / sqrtf(sk + 1e-6f);
#pragma unroll
                for (int i = 0; i < 8; ++i) { xq[i] *= iq; xk[i] *= ik; }
            }
            float xa[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                xa[i] = r < L ? expf(kGated ? gate_decay(xg[i], dtb[i], lamneg) : xg[i]) : 1.f;
            st4s(&sm.q[r][c0], make_float4(xq[0], xq[1], xq[2], xq[3]));
            st4s(&sm.q[r][c0 + 4], make_float4(xq[4], xq[5], xq[6], xq[7]));
            st4s(&sm.k[r][c0], make_float4(xk[0], xk[1], xk[2], xk[3]));
            st4s(&sm.k[r][c0 + 4], make_float4(xk[4], xk[5], xk[6], xk[7]));
            st4s(&sm.a[r][c0], make_float4(xa[0], xa[1], xa[2], xa[3]));
            st4s(&sm.a[r][c0 + 4], make_float4(xa[4], xa[5], xa[6], xa[7]));
            st4s(&sm.v[r][c0], make_float4(xv[0], xv[1], xv[2], xv[3]));
            st4s(&sm.v[r][c0 + 4], make_float4(xv[4], xv[5], xv[6], xv[7]));
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
    }
    __syncthreads();

    // ---- 2. pairs inside each 4-token sub-block: 16 lanes per sub-block, each
    // with 8 channels (c0 .. c0+3 and c0+64 .. c0+67); the 10 q.k and 6 k.k
    // partial sums of a sub-block are reduce-scattered over its 16 lanes
    {
        const int r0 = (tid >> 4) * S4, c0 = (tid & 15) * 4;
        float4 qa[S4][2], ka[S4][2], aa[S4][2];
#pragma unroll
        for (int u = 0; u < S4; ++u)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                qa[u][hh] = ld4s(&sm.q[r0 + u][c0 + 64 * hh]);
                ka[u][hh] = ld4s(&sm.k[r0 + u][c0 + 64 * hh]);
                aa[u][hh] = ld4s(&sm.a[r0 + u][c0 + 64 * hh]);
            }
        // entries 0..9: q.k for (i, j) = (0,0) (1,0) (2,0) (3,0) (1,1) (2,1) (3,1)
        // (2,2) (3,2) (3,3); 10..15: k.k for (1,0) (2,0) (3,0) (2,1) (3,1) (3,2)
        float val[16];
        int nq = 0, nk = 10;
#pragma unroll
        for (int j = 0; j < S4; ++j) {
            float4 kp0 = ka[j][0], kp1 = ka[j][1];
#pragma unroll
            for (int i = j; i < S4; ++i) {
                if (i > j) {
                    kp0 = mul4(kp0, aa[i][0]);
                    kp1 = mul4(kp1, aa[i][1]);
                    val[nk++] = dot4(ka[i][1], kp1, dot4(ka[i][0], kp0, 0.f));
                }
                val[nq++] = dot4(qa[i][1], kp1, dot4(qa[i][0], kp0, 0.f));
            }
        }
        ReduceScatter<16, 8>::run(val, lane);
        const int e = lane & 15;
        // (i, j) of entry e, two bits each
        constexpr uint32_t I_OF = (0u << 0) | (1u << 2) | (2u << 4) | (3u << 6) | (1u << 8) |
                                  (2u << 10) | (3u << 12) | (2u << 14) | (3u << 16) | (3u << 18) |
                                  (1u << 20) | (2u << 22) | (3u << 24) | (2u << 26) | (3u << 28) |
                                  (3u << 30);
        constexpr uint32_t J_OF = (0u << 0) | (0u << 2) | (0u << 4) | (0u << 6) | (1u << 8) |
                                  (1u << 10) | (1u << 12) | (2u << 14) | (2u << 16) | (3u << 18) |
                                  (0u << 20) | (0u << 22) | (0u << 24) | (1u << 26) | (1u << 28) |
                                  (2u << 30);
        const int i = r0 + (int)((I_OF >> (2 * e)) & 3u), j = r0 + (int)((J_OF >> (2 * e)) & 3u);
        if (e < 10) sm.aqk[i][j] = val[0];
        else sm.akk[i][j] = sm.beta[i] * val[0];
    }
    __syncthreads();

    // ---- 3. per (16-token block, channel): fwd4 / bwd4 inside each sub-block,
    // the sub-block totals and the block total; q^ -> Qf4, k^ -> Kf4, e^g -> Kb4
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
        const int I = (tid >> 7) + 2 * ii, c = tid & 127;
        float bt = 1.f;
#pragma unroll
        for (int s = 0; s < SB / S4; ++s) {
            const int r0 = I * SB + s * S4;
            float av[S4], kv[S4];
#pragma unroll
            for (int u = 0; u < S4; ++u) { av[u] = sm.a[r0 + u][c]; kv[u] = sm.k[r0 + u][c]; }
            float p = 1.f;
#pragma unroll
            for (int u = 0; u < S4; ++u) {
                p *= av[u];
                sm.q[r0 + u][c] *= p;
                sm.k[r0 + u][c] = kv[u] * p;
            }
            float pb = 1.f;
#pragma unroll
            for (int u = S4 - 1; u >= 0; --u) {
                sm.a[r0 + u][c] = kv[u] * pb;
                pb *= av[u];
            }
            sm.t4[I * (SB / S4) + s][c] = p;
            bt *= p;
        }
        sm.blk[I][c] = bt;
        const float t1 = sm.t4[I * (SB / S4) + 1][c], t2 = sm.t4[I * (SB / S4) + 2][c];
        sm.mid4[I][0][c] = 1.f;
        sm.mid4[I][1][c] = t1;
        sm.mid4[I][2][c] = t2;
        sm.mid4[I][3][c] = t1 * t2;
    }
    __syncthreads();

    // ---- 4. pairs in different sub-blocks of one 16-token block: 24 tiles of
    // 4 x 4, eight lanes per tile (a quarter warp, so that the lanes of a tile
    // read the same Kb4 rows at once), each lane one row of A_kk or of A_qk.
    // Threads 0..191 sum channels 0..95 of their row; threads 192..255 sum
    // channels 96..127 of three rows each and hand those partial sums over
    // through the (not yet used) T array.
    {
        auto row_of = [&](int tl, int& i, int& rj, const float*& midp) {
            const int tile = tl >> 3, I = tile / 6, pr = tile % 6;
            const int sa = pr == 0 ? 1 : (pr < 3 ? 2 : 3);      // (sa, sb): (1,0) (2,0) (2,1)
            const int sb = pr == 0 ? 0 : (pr < 3 ? pr - 1 : pr - 3);   //   (3,0) (3,1) (3,2)
            i = I * SB + sa * S4 + ((tl >> 1) & 3);
            rj = I * SB + sb * S4;
            // sub-blocks strictly between: none, 1, 2 or 1 and 2
            midp = &sm.mid4[I][sa - sb == 1 ? 0 : (sa - sb == 3 ? 3 : sb + 1)][0];
        };
        float acc[S4];
        auto row_sums = [&](int tl, int c0, int c1) {
            int i, rj;
            const float* midp;
            row_of(tl, i, rj, midp);
            const float* x = (tl & 1) ? &sm.q[i][0] : &sm.k[i][0];
#pragma unroll
            for (int u = 0; u < S4; ++u) acc[u] = 0.f;
#pragma unroll 4
            for (int c = c0; c < c1; c += 4) {
                const float4 mid = ld4s(midp + c);
                const float4 xv = ld4s(x + c);
#pragma unroll
                for (int u = 0; u < S4; ++u) acc[u] = dot4(xv, mul4(ld4s(&sm.a[rj + u][c]), mid), acc[u]);
            }
        };
        float* part = &sm.tf[0][0];                         // [192 rows][4]
        if (tid >= 24 * 8) {
#pragma unroll 1
            for (int k3 = 0; k3 < 3; ++k3) {
                const int tl = tid - 24 * 8 + 64 * k3;
                row_sums(tl, 96, DK);
                st4s(part + tl * 4, make_float4(acc[0], acc[1], acc[2], acc[3]));
            }
        } else {
            row_sums(tid, 0, 96);
        }
        __syncthreads();
        if (tid < 24 * 8) {
            int i, rj;
            const float* midp;
            row_of(tid, i, rj, midp);
            const float4 pp = ld4s(part + tid * 4);
            const bool qk = tid & 1;
            const float sc = qk ? 1.f : sm.beta[i];
            st4s(qk ? &sm.aqk[i][rj] : &sm.akk[i][rj],
                 make_float4(sc * (acc[0] + pp.x), sc * (acc[1] + pp.y), sc * (acc[2] + pp.z),
                             sc * (acc[3] + pp.w)));
        }
    }
    __syncthreads();

    // ---- 5. 4-token factors -> 16-token factors: Qf16 = Qf4 o (sub-blocks
    // before it in the block), Kf16 likewise, Kb16 = Kb4 o (sub-blocks after it)
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
        const int I = (tid >> 7) + 2 * ii, c = tid & 127;
        float t[SB / S4];
#pragma unroll
        for (int s = 0; s < SB / S4; ++s) t[s] = sm.t4[I * (SB / S4) + s][c];
        if (ii == 0) {
            const float b0 = sm.blk[0][c], b1 = sm.blk[1][c], b2 = sm.blk[2][c], b3 = sm.blk[3][c];
            if (tid < 128) {
                sm.mid16[0][c] = 1.f;
                sm.mid16[1][c] = b1;
                sm.pre16[0][c] = 1.f;
                sm.pre16[1][c] = b0;
                sm.pre16[2][c] = b0 * b1;
                sm.pre16[3][c] = b0 * b1 * b2;
            } else {
                sm.mid16[2][c] = b2;
                sm.mid16[3][c] = b1 * b2;
                sm.post16[0][c] = b1 * b2 * b3;
                sm.post16[1][c] = b2 * b3;
                sm.post16[2][c] = b3;
                sm.post16[3][c] = 1.f;
            }
        }
        const float pre[4] = {1.f, t[0], t[0] * t[1], t[0] * t[1] * t[2]};
        const float post[4] = {t[1] * t[2] * t[3], t[2] * t[3], t[3], 1.f};
#pragma unroll
        for (int s = 0; s < SB / S4; ++s)
#pragma unroll
            for (int u = 0; u < S4; ++u) {
                const int r = I * SB + s * S4 + u;
                sm.q[r][c] *= pre[s];
                sm.k[r][c] *= pre[s];
                sm.a[r][c] *= post[s];
            }
    }
    __syncthreads();

    // ---- 6. pairs in different 16-token blocks: one warp per block pair, each
    // lane a 2 x 4 tile of A_kk and of A_qk (rows r and r + 8: the eight lanes
    // of a quarter warp read eight consecutive rows and one set of Kb16 rows).
    // Warps 0..5 sum channels 0..95 of their pair; warps 6 and 7 sum channels
    // 96..127 of three pairs each and hand those partial sums over through the
    // (not yet used) T array, so that every warp runs 96 channel steps.
    {
        float skk[2][4], sqk[2][4];
        auto tile_sums = [&](int pr, int c0, int c1) {
            const int I = pr == 0 ? 1 : (pr < 3 ? 2 : 3);        // (I, J): (1,0) (2,0) (2,1)
            const int J = pr == 0 ? 0 : (pr < 3 ? pr - 1 : pr - 3);   //   (3,0) (3,1) (3,2)
            const int ib = I * SB + (lane & 7), j0 = J * SB + (lane >> 3) * 4;
            // blocks strictly between: none, 1, 2 or 1 and 2
            const float* midp = &sm.mid16[I - J == 1 ? 0 : (I - J == 3 ? 3 : J + 1)][0];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int x = 0; x < 4; ++x) { skk[r][x] = 0.f; sqk[r][x] = 0.f; }
#pragma unroll 2
            for (int c = c0; c < c1; c += 4) {
                const float4 mid = ld4s(midp + c);
                float4 kb[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) kb[u] = mul4(ld4s(&sm.a[j0 + u][c]), mid);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float4 kf = ld4s(&sm.k[ib + 8 * r][c]), qf = ld4s(&sm.q[ib + 8 * r][c]);
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        skk[r][x] = dot4(kf, kb[x], skk[r][x]);
                        sqk[r][x] = dot4(qf, kb[x], sqk[r][x]);
                    }
                }
            }
        };
        float* part = &sm.tf[0][0];                         // [pair][16 sums][32 lanes]
        if (warp >= 6) {
#pragma unroll 1
            for (int p3 = 0; p3 < 3; ++p3) {
                const int pr = 3 * (warp - 6) + p3;
                tile_sums(pr, 96, DK);
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        part[(pr * 16 + 4 * r + x) * 32 + lane] = skk[r][x];
                        part[(pr * 16 + 8 + 4 * r + x) * 32 + lane] = sqk[r][x];
                    }
            }
        } else {
            tile_sums(warp, 0, 96);
        }
        __syncthreads();
        if (warp < 6) {
            const int pr = warp;
            const int I = pr == 0 ? 1 : (pr < 3 ? 2 : 3);
            const int J = pr == 0 ? 0 : (pr < 3 ? pr - 1 : pr - 3);
            const int ib = I * SB + (lane & 7), j0 = J * SB + (lane >> 3) * 4;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    skk[r][x] += part[(pr * 16 + 4 * r + x) * 32 + lane];
                    sqk[r][x] += part[(pr * 16 + 8 + 4 * r + x) * 32 + lane];
                }
                const float b = sm.beta[ib + 8 * r];
                st4s(&sm.akk[ib + 8 * r][j0],
                     make_float4(b * skk[r][0], b * skk[r][1], b * skk[r][2], b * skk[r][3]));
                st4s(&sm.aqk[ib + 8 * r][j0], make_float4(sqk[r][0], sqk[r][1], sqk[r][2], sqk[r][3]));
            }
        }
    }
    __syncthreads();

    // ---- 7. X = beta k^ o e^G (in place of Kf16) and beta v; Q' = q^ o e^G
    // (rows 64.. of the [W; Q'] operand), K'' = k^ o e^{G_last - G} and A_qk
    // (zero above the diagonal) to the record as FP16 pairs (|x| <= 1, scale
    // 1); d = e^{G_last}
#pragma unroll 2
    for (int m = 0; m < C * DK / 8 / NT; ++m) {
        const int e = tid + NT * m, r = e >> 4, c = (e & 15) * 8, I = r / SB;
        const float b = sm.beta[r];
        float qv[8], kv[8];
#pragma unroll
        for (int hx = 0; hx < 2; ++hx) {
            const int cx = c + 4 * hx;
            const float4 pre = ld4s(&sm.pre16[I][cx]), post = ld4s(&sm.post16[I][cx]);
            st4s(&sm.k[r][cx], scale4(mul4(ld4s(&sm.k[r][cx]), pre), b));
            st4s(&sm.v[r][cx], scale4(ld4s(&sm.v[r][cx]), b));
            const float4 q4 = mul4(ld4s(&sm.q[r][cx]), pre), k4 = mul4(ld4s(&sm.a[r][cx]), post);
            qv[4 * hx] = q4.x; qv[4 * hx + 1] = q4.y; qv[4 * hx + 2] = q4.z; qv[4 * hx + 3] = q4.w;
            kv[4 * hx] = k4.x; kv[4 * hx + 1] = k4.y; kv[4 * hx + 2] = k4.z; kv[4 * hx + 3] = k4.w;
        }
        st8_pair(recb + R_WQ, R_WQ_LO - R_WQ, 16384, 64 + r, c, qv, 1.f);
        st8_pair(recb + R_LATE + L_KT, L_KT_LO - L_KT, 8192, r, c, kv, 1.f);
    }
#pragma unroll
    for (int m = 0; m < C * C / 8 / NT; ++m) {
        const int e = tid + NT * m, r = e >> 3, j = (e & 7) * 8;
        const float4 x0 = ld4s(&sm.aqk[r][j]), x1 = ld4s(&sm.aqk[r][j + 4]);
        const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float y[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) y[u] = j + u <= r ? x[u] : 0.f;
        st8_pair(recb + R_LATE + L_AQK, L_AQK_LO - L_AQK, 0, r, j, y, 1.f);
    }
    if (tid < DK / 4) {
        const int c = tid * 4;
        st4s(reinterpret_cast<float*>(recb + R_LATE + L_DEC) + c,
             mul4(ld4s(&sm.pre16[NB - 1][c]), ld4s(&sm.blk[NB - 1][c])));
    }
    __syncthreads();

    // ---- 8. T = (I + A_kk)^-1 (blocked; unit diagonal, read as lower triangular)
    chunk_ops::chunk_inverse_f32(sm.akk, sm.tf, tid, warp, lane);

    // ---- 9. W = T X (threads 0..127) and U = T (beta V) (threads 128..255):
    // each thread a 4 x 8 tile for row groups g and 15 - g in turn, so that
    // every thread runs the same number of steps over the triangle of T
    {
        const int tt = tid & 127, gp = tt >> 4, c0 = (tt & 15) * 8;
        const float (*src)[LDK] = tid < 128 ? sm.k : sm.v;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int i0 = 4 * (pass ? 15 - gp : gp);
            float w[4][8];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int x = 0; x < 8; ++x) w[r][x] = 0.f;
            for (int kk = 0; kk < i0; kk += 4) {           // the full blocks left of the diagonal
                float4 t4[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) t4[r] = ld4s(&sm.tf[i0 + r][kk]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 xa = ld4s(&src[kk + e][c0]), xb = ld4s(&src[kk + e][c0 + 4]);
                    const float xs[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float t = f4at(t4[r], e);
#pragma unroll
                        for (int x = 0; x < 8; ++x) w[r][x] = fmaf(t, xs[x], w[r][x]);
                    }
                }
            }
            {
                // the diagonal block: T is lower triangular with a unit diagonal,
                // and its entries above the diagonal (scratch of the merges) count as 0
                float4 t4[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) t4[r] = ld4s(&sm.tf[i0 + r][i0]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 xa = ld4s(&src[i0 + e][c0]), xb = ld4s(&src[i0 + e][c0 + 4]);
                    const float xs[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                    for (int r = e; r < 4; ++r) {
                        const float t = r == e ? 1.f : f4at(t4[r], e);
#pragma unroll
                        for (int x = 0; x < 8; ++x) w[r][x] = fmaf(t, xs[x], w[r][x]);
                    }
                }
            }
            if (tid < 128) {
                // W rows as FP16 pairs, row i scaled by s_i from the row's largest
                // magnitude (over the 16 lanes of a half warp that hold the row)
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    float mx = 0.f;
#pragma unroll
                    for (int x = 0; x < 8; ++x) mx = fmaxf(mx, fabsf(w[r][x]));
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    float sc, inv;
                    pow2_scale(mx, sc, inv);
                    st8_pair(recb + R_WQ, R_WQ_LO - R_WQ, 16384, i0 + r, c0, w[r], sc);
                    if ((tt & 15) == 0) reinterpret_cast<float*>(recb + R_WINV)[i0 + r] = inv;
                }
            } else {
                // U rows in FP32, V halves apart, 16-byte pieces swizzled by row
                unsigned char* uh = recb + R_U + (c0 >> 6) * R_UHALF;
                const int p0 = (c0 & 63) >> 2;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = i0 + r;
                    st4s(reinterpret_cast<float*>(uh + i * 256 + ((p0 ^ (i & 7)) << 4)),
                         make_float4(w[r][0], w[r][1], w[r][2], w[r][3]));
                    st4s(reinterpret_cast<float*>(uh + i * 256 + (((p0 + 1) ^ (i & 7)) << 4)),
                         make_float4(w[r][4], w[r][5], w[r][6], w[r][7]));
                }
            }
        }
    }
}

// ---------------------------------------------------------------- scan
// One CTA per (sequence, head, half of V): eight epilogue warps and one
// control warp whose lane 0 issues the bulk copies and the MMAs.  Epilogue
// thread (quad q = warp & 3, half hf = warp >> 2, lane l) owns TMEM lane
// row = 32 q + l and columns 32 hf .. 32 hf + 31 of this CTA's 64: the FP32
// state S[row][v] for those columns lives in its registers.  Per chunk c, in
// TMEM region R = 256 (c & 1):
//   control:  D1 = [W s; Q'] (S sS) (24 MMAs, M = 128, K = 128 channels: rows
//             0..63 W S, 64..127 Q' S), commit d1_done
//   Delta warps (lanes 0..63): Delta = U - D1 / (s_i sS); its largest
//             magnitude over the four warps gives sD; Delta sD as FP16 pairs
//             to shared memory; arrive delta_ready
//   control:  the next chunk's early part may come; P = K''^T (Delta sD) and
//             O2 = [any; A_qk] (Delta sD) (12 MMAs each, K = 64 tokens; rows
//             0..63 of O2's A operand are the 8 KiB before A_qk, finite
//             values whose products land in rows that are never read)
//   all warps: S <- Diag(d) S + P / sD; the new state's largest magnitude over
//             the eight warps gives the next sS; S sS as FP16 pairs; arrive
//             s_ready
//   O warps (lanes 64..127): O = D1 / sS + O2 / sD once o_done has come,
//             arrive o_read, store the chunk's output rows
// The record comes in three copies, each into one region of shared memory:
// the [W; Q'] pairs once D1's MMAs are complete, U and 1/s_i once the Delta
// warps have read them, the late part once chunk c - 1's P, O2 and Diag(d) S
// are done.
constexpr int VH = 64;
constexpr int SCAN_THREADS = NT + 32;
constexpr int kL2Ahead = 4;                   // records prefetched into L2 this many chunks ahead
constexpr uint32_t kEpiBar = 1;               // named barrier of the 256 epilogue threads
constexpr uint32_t kDeltaBar = 2;             // named barrier of the four Delta warps
constexpr uint32_t F_E = 0;                   // early part: [W; Q'] pairs, 1/s_i
constexpr uint32_t F_U = R_U;                 //             U of this half of V [64 i][64 v]
constexpr uint32_t F_L = 82944;               // late part (1 KiB aligned)
constexpr uint32_t F_S = F_L + 50176;         // S sS pair: MN-major [128 c][64 v] fp16, lo 16 KiB after
constexpr uint32_t F_D = F_S + 32768;         // Delta sD pair: MN-major [64 i][64 v], lo 8 KiB after
constexpr uint32_t F_BAR = F_D + 16384;       // 10 mbarriers, TMEM slot, abort flag, maxima, 1/sD
constexpr uint32_t F_SMEM = F_BAR + 256 + 1024;
static_assert(F_U + R_UHALF <= F_L && F_L % 1024 == 0 && F_L + R_LATE_BYTES <= F_S, "scan regions");
static_assert(F_S % 1024 == 0 && F_D % 1024 == 0 && F_SMEM <= 232448, "FP32 scan shared memory");
constexpr uint32_t F_TM_D1 = 0, F_TM_P = 64, F_TM_O2 = 128, F_TM_REGION = 256, F_TM_COLS = 512;

__device__ __forceinline__ void store_row32(float* p, const float (&o)[32])
{
#pragma unroll
    for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(p)[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
}
__device__ __forceinline__ void store_row32(__nv_bfloat16* p, const float (&o)[32])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[8 * q + 2 * e], o[8 * q + 2 * e + 1]);
            w[e] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        reinterpret_cast<uint4*>(p)[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

template <typename TOut>
__global__ void __launch_bounds__(SCAN_THREADS, 1) fp32_scan_kernel(ChunkArgs args,
                                                                    const int32_t* __restrict__ hdr,
                                                                    const unsigned char* __restrict__ records)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];   // aligned to 1 KiB below
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    unsigned char* sm = smem_raw + pad;
    const uint32_t sb = raw_s + pad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool ctrl = warp == NT / 32;
    const int quad = warp & 3, half = (warp >> 2) & 1;
    const int row = 32 * quad + lane;                      // TMEM lane
    const bool dwarp = quad < 2;                           // lanes 0..63: W S rows -> Delta
    const int H = args.H;
    const int vh = blockIdx.x & 1, hb = blockIdx.x >> 1;
    const int n = hdr[kPlanOffsets + args.N + 1 + hb / H], h = hb % H;
    const int bos = args.cu_seqlens[n], eos = args.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || (int64_t)eos > args.T) return;   // reported by the plan
    const int nch = (eos - bos + C - 1) / C;
    if (hdr[kPlanOffsets + n] + nch > split_chunk_bound(args.N, args.T)) return;   // bad offsets elsewhere
    const unsigned char* rec0 =
        records + ((int64_t)hdr[kPlanOffsets + n] * H + h) * (int64_t)R_BYTES;
    const int64_t rstride = (int64_t)H * R_BYTES;
    TOut* __restrict__ out = static_cast<TOut*>(args.out);
    const int v0 = VH * vh + 32 * half;                    // this thread's first column of V
    // [0] [W; Q'] pairs, [1] late part, [2] d1_done, [3] p_done, [4]
    // delta_ready (128), [5] s_ready (NT), [6] drain after a failure, [7]
    // o_done, [8,9] o_read of even and odd chunks (128), [10] U and 1/s_i
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + F_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + F_BAR + 96);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(sm + F_BAR + 100);
    float* smax = reinterpret_cast<float*>(sm + F_BAR + 128);     // [2][8]: state maxima by warp
    float* dmax = reinterpret_cast<float*>(sm + F_BAR + 192);     // [2][4]: Delta maxima by warp
    float* dinv = reinterpret_cast<float*>(sm + F_BAR + 224);     // [2]: 1/sD by chunk parity

    // The largest |x| over the 256 epilogue threads (exchange `k`, parity-alternating slots).
    auto epi_max = [&](float mx, int k) -> float {
        mx = warp_max(mx);
        float* slot = smax + 8 * (k & 1);
        if (lane == 0) slot[warp] = mx;
        named_sync(kEpiBar, NT);
        const float4 a = reinterpret_cast<const float4*>(slot)[0], b = reinterpret_cast<const float4*>(slot)[1];
        return fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)), fmaxf(fmaxf(b.x, b.y), fmaxf(b.z, b.w)));
    };

    // ---- the entering state: S[row][v0 .. v0 + 31], and its scaled pair
    float S[32];
    float s_S = 1.f, inv_S = 1.f;                          // scale of the state's copy
    if (!ctrl) {
        if (args.initial_state != nullptr) {
            const float4* s0 = reinterpret_cast<const float4*>(
                args.initial_state + (((int64_t)n * H + h) * DK + row) * DV + v0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = s0[q];
                S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) S[u] = 0.f;
        }
        float mx = 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) mx = fmaxf(mx, fabsf(S[u]));
        pow2_scale(epi_max(mx, 1), s_S, inv_S);
#pragma unroll
        for (int q = 0; q < 4; ++q) st8_pair(sm + F_S, 16384, 0, row, 32 * half + 8 * q, S + 8 * q, s_S);
    }
    if (warp == 0) {
        tmem_alloc(tslot, F_TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 11; ++b)
            mbar_init(&bar[b], (b == 4 || b == 8 || b == 9) ? NT / 2 : b == 5 ? NT : 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tlane = tmem + ((uint32_t)(32 * quad) << 16);

    auto wait_or_abort = [&](uint64_t* m, uint32_t parity) -> bool {
        for (uint32_t j = 0; j < kPollsPerCheck; ++j)
            if (mbar_try_wait(m, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t i = 0; i < kMaxTimerChecks; ++i) {
            for (uint32_t j = 0; j < kPollsPerCheck; ++j)
                if (mbar_try_wait(m, parity)) return true;
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
        *abort_flag = 1;
        return false;
    };

    if (ctrl) {
        if (lane == 0) {
            // the early part in two copies: [W; Q'] once D1 has read the last
            // one, U and 1/s_i once the Delta warps have
            auto issue_wq = [&](int c) {
                mbar_arrive_expect_tx(&bar[0], R_WINV);
                bulk_g2s(sm + F_E, rec0 + c * rstride, R_WINV, &bar[0]);
            };
            auto issue_u = [&](int c) {
                const unsigned char* r = rec0 + c * rstride;
                mbar_arrive_expect_tx(&bar[10], (R_U - R_WINV) + R_UHALF);
                bulk_g2s(sm + F_E + R_WINV, r + R_WINV, R_U - R_WINV, &bar[10]);
                bulk_g2s(sm + F_U, r + R_U + vh * R_UHALF, R_UHALF, &bar[10]);
            };
            auto issue_late = [&](int c) {
                mbar_arrive_expect_tx(&bar[1], R_LATE_BYTES);
                bulk_g2s(sm + F_L, rec0 + c * rstride + R_LATE, R_LATE_BYTES, &bar[1]);
            };
            // copies issued (at most one of each part in flight)
            int w_issued = 0, u_issued = 0, l_issued = 0, c = 0;
            if (nch > 0) {
                issue_wq(0);
                issue_u(0);
                issue_late(0);
                w_issued = u_issued = l_issued = 1;
            }
            for (int cc = 1; cc < min(kL2Ahead, nch); ++cc) bulk_prefetch_l2(rec0 + cc * rstride, R_BYTES);
            bool fail = false, any_mma = false;
            constexpr uint32_t id_d1 = idesc(kFmtF16, 128, VH, false, true);
            constexpr uint32_t id_p = idesc(kFmtF16, 128, VH, true, true);
            constexpr uint32_t id_o = idesc(kFmtF16, 128, VH, false, true);
            // operand descriptors at k-step 0, computed once (every region is fixed)
            const uint64_t dWh = desc_kmajor(sb + F_E + R_WQ, 128, 0);
            const uint64_t dWl = desc_kmajor(sb + F_E + R_WQ_LO, 128, 0);
            const uint64_t dSh = desc_mnmajor64(sb + F_S, 0), dSl = desc_mnmajor64(sb + F_S + 16384, 0);
            const uint64_t dKh = desc_mnmajor128(sb + F_L + L_KT, 8192, 0);
            const uint64_t dKl = desc_mnmajor128(sb + F_L + L_KT_LO, 8192, 0);
            const uint64_t dAh = desc_kmajor(sb + F_L + L_AQK - 8192, 128, 0);
            const uint64_t dAl = desc_kmajor(sb + F_L + L_AQK_LO - 8192, 128, 0);
            const uint64_t dDh = desc_mnmajor64(sb + F_D, 0), dDl = desc_mnmajor64(sb + F_D + 8192, 0);
            for (; c < nch; ++c) {
                const uint32_t R = tmem + F_TM_REGION * (c & 1);
                if (c > 0) {
                    // chunk c - 1's state is current, and its P, O2 and d are done
                    // with the late region
                    if (!wait_or_abort(&bar[5], (c - 1) & 1) || !wait_or_abort(&bar[7], (c - 1) & 1)) {
                        fail = true;
                        break;
                    }
                    issue_late(c);
                    ++l_issued;
                }
                // chunk c - 2's O has left region (c & 1)
                if (c > 1 && !wait_or_abort(&bar[8 + (c & 1)], ((c - 2) >> 1) & 1)) { fail = true; break; }
                if (!wait_or_abort(&bar[0], c & 1)) { fail = true; break; }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint64_t ah = desc_advance(dWh, kmajor_off(128, s));
                    const uint64_t al = desc_advance(dWl, kmajor_off(128, s));
                    const uint64_t bh = desc_advance(dSh, mnmajor_off(s)), bl = desc_advance(dSl, mnmajor_off(s));
                    mma_f16(R + F_TM_D1, ah, bh, id_d1, s > 0);
                    mma_f16(R + F_TM_D1, ah, bl, id_d1, 1);
                    mma_f16(R + F_TM_D1, al, bh, id_d1, 1);
                }
                commit(&bar[2]);
                any_mma = true;
                if (c + kL2Ahead < nch) bulk_prefetch_l2(rec0 + (c + kL2Ahead) * rstride, R_BYTES);
                if (c + 1 < nch) {
                    // D1's MMAs are complete: the next [W; Q'] may come
                    if (!wait_or_abort(&bar[2], c & 1)) { fail = true; break; }
                    issue_wq(c + 1);
                    ++w_issued;
                }
                if (!wait_or_abort(&bar[4], c & 1)) { fail = true; break; }
                // the Delta warps have read U and 1/s_i
                if (c + 1 < nch) {
                    issue_u(c + 1);
                    ++u_issued;
                }
                if (!wait_or_abort(&bar[1], c & 1)) { fail = true; break; }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_advance(dKh, mnmajor_off(s));
                    const uint64_t al = desc_advance(dKl, mnmajor_off(s));
                    const uint64_t bh = desc_advance(dDh, mnmajor_off(s)), bl = desc_advance(dDl, mnmajor_off(s));
                    mma_f16(R + F_TM_P, ah, bh, id_p, s > 0);
                    mma_f16(R + F_TM_P, ah, bl, id_p, 1);
                    mma_f16(R + F_TM_P, al, bh, id_p, 1);
                }
                commit(&bar[3]);
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ah = desc_advance(dAh, kmajor_off(128, s));
                    const uint64_t al = desc_advance(dAl, kmajor_off(128, s));
                    const uint64_t bh = desc_advance(dDh, mnmajor_off(s)), bl = desc_advance(dDl, mnmajor_off(s));
                    mma_f16(R + F_TM_O2, ah, bh, id_o, s > 0);
                    mma_f16(R + F_TM_O2, ah, bl, id_o, 1);
                    mma_f16(R + F_TM_O2, al, bh, id_o, 1);
                }
                commit(&bar[7]);
            }
            if (fail) {
                *abort_flag = 1;
                report_status(args.status, KDA_ERR_TIMEOUT);
                // the MMAs and copies in flight finish before the CTA leaves
                if (any_mma) {
                    commit(&bar[6]);
                    mbar_wait(&bar[6], 0);
                }
                // the last copy of each part has landed (no later one was issued)
                if (w_issued > 0) mbar_wait(&bar[0], (w_issued - 1) & 1);
                if (u_issued > 0) mbar_wait(&bar[10], (u_issued - 1) & 1);
                if (l_issued > 0) mbar_wait(&bar[1], (l_issued - 1) & 1);
            }
        }
    } else {
        float nan_acc = 0.f;
        // test hook: CTA 0 withholds its first delta_ready arrival
        const bool withhold = args.fault == KDA_TEST_FAULT_SCAN && blockIdx.x == 0;
        bool fail = false;
        const float* winv = reinterpret_cast<const float*>(sm + F_E + R_WINV);
        const float* dec = reinterpret_cast<const float*>(sm + F_L + L_DEC);
        for (int c = 0; c < nch; ++c) {
            const uint32_t R = tlane + F_TM_REGION * (c & 1);
            {
                // (an O warp that gave up on the previous chunk carries `fail` here)
                const bool ok = !fail && (!dwarp || wait_or_abort(&bar[10], c & 1));
                if (named_sync_or(kEpiBar, NT, !ok)) { fail = true; break; }
            }
            if (dwarp) {
                // U[i][v0 .. v0 + 31] (i = row), read while D1 runs
                float u[32];
                const unsigned char* up = sm + F_U + row * 256;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int p = 8 * half + q;
                    const float4 x = *reinterpret_cast<const float4*>(up + ((p ^ (row & 7)) << 4));
                    u[4 * q] = x.x; u[4 * q + 1] = x.y; u[4 * q + 2] = x.z; u[4 * q + 3] = x.w;
                }
                const float wsc = winv[row] * inv_S;
                const bool ok = wait_or_abort(&bar[2], c & 1);
                if (named_sync_or(kDeltaBar, NT / 2, !ok)) {
                    fail = true;                           // the others see the abort flag
                } else {
                    fence_after_sync();
                    // Delta = U - W S; then its pair at scale sD
                    float ws[32];
                    tmem_ld32(R + F_TM_D1 + 32 * half, ws);
                    float mx = 0.f;
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        u[x] = fmaf(-ws[x], wsc, u[x]);
                        mx = fmaxf(mx, fabsf(u[x]));
                    }
                    mx = warp_max(mx);
                    float* slot = dmax + 4 * (c & 1);
                    if (lane == 0) slot[quad + 2 * half] = mx;
                    named_sync(kDeltaBar, NT / 2);
                    const float4 m4 = *reinterpret_cast<const float4*>(slot);
                    float s_D, inv_D;
                    pow2_scale(fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w)), s_D, inv_D);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st8_pair(sm + F_D, 8192, 0, row, 32 * half + 8 * q, u + 8 * q, s_D);
                    if (tid == 0) dinv[c & 1] = inv_D;
                    fence_async_smem();
                    fence_before_sync();
                    if (!(withhold && c == 0)) mbar_arrive(&bar[4]);
                }
            }
            {
                const bool ok = !fail && wait_or_abort(&bar[3], c & 1) && wait_or_abort(&bar[1], c & 1);
                if (named_sync_or(kEpiBar, NT, !ok)) { fail = true; break; }
            }
            fence_after_sync();
            const float inv_D = dinv[c & 1];
            const float inv_S_used = inv_S;                // the scale of this chunk's D1
            {
                // S <- Diag(d) S + P / sD; the new state's pair at its own scale
                const float dc = dec[row];
                float p[32];
                tmem_ld32(R + F_TM_P + 32 * half, p);
                float mx = 0.f;
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    S[u] = fmaf(S[u], dc, p[u] * inv_D);
                    mx = fmaxf(mx, fabsf(S[u]));
                }
                pow2_scale(epi_max(mx, c), s_S, inv_S);
#pragma unroll
                for (int q = 0; q < 4; ++q) st8_pair(sm + F_S, 16384, 0, row, 32 * half + 8 * q, S + 8 * q, s_S);
            }
            fence_async_smem();
            fence_before_sync();
            mbar_arrive(&bar[5]);
            if (!dwarp) {
                // O rows (token i = row - 64) leave TMEM, then go out from registers
                const bool ok = wait_or_abort(&bar[7], c & 1);
                if (ok) {
                    fence_after_sync();
                    float o[32], o2[32];
                    tmem_ld32x2(R + F_TM_D1 + 32 * half, R + F_TM_O2 + 32 * half, o, o2);
                    fence_before_sync();
                    mbar_arrive(&bar[8 + (c & 1)]);
                    const int i = row - 64, t = bos + c * C + i;
                    if (t < eos) {
                        TOut* op = out + ((int64_t)t * H + h) * DV + v0;
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            o[u] = args.scale * fmaf(o[u], inv_S_used, o2[u] * inv_D);
                            nan_acc = fmaf(o[u], 0.f, nan_acc);
                        }
                        store_row32(op, o);
                    }
                } else {
                    fail = true;                           // seen at the next chunk's barrier
                }
            }
        }
        if (fail) {
            *abort_flag = 1;
            if (tid == 0) report_status(args.status, KDA_ERR_TIMEOUT);
        } else if (args.final_state != nullptr) {
            float4* fs = reinterpret_cast<float4*>(args.final_state + (((int64_t)n * H + h) * DK + row) * DV + v0);
#pragma unroll
            for (int u = 0; u < 32; ++u) nan_acc = fmaf(S[u], 0.f, nan_acc);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                fs[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
        }
        if (nan_acc != nan_acc) report_status(args.status, KDA_ERR_RANGE);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, F_TM_COLS);
}

template <typename TIn, int kGate>
cudaError_t launch_prep_typed(const ChunkArgs& a, const int32_t* hdr, unsigned char* rec,
                              int64_t units, cudaStream_t stream)
{
    auto kern = fp32_prep_kernel<TIn, kGate>;
    const int smem = (int)sizeof(PrepSmem);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)units, NT, smem, stream>>>(a, hdr, rec);
    return cudaGetLastError();
}

template <int kGate>
cudaError_t launch_prep_gate(const ChunkArgs& a, const int32_t* hdr, unsigned char* rec,
                             int64_t units, cudaStream_t stream)
{
    return a.qkv_bf16 ? launch_prep_typed<__nv_bfloat16, kGate>(a, hdr, rec, units, stream)
                      : launch_prep_typed<float, kGate>(a, hdr, rec, units, stream);
}

}  // namespace

int64_t fp32_split_workspace_bytes(int32_t N, int64_t T, int32_t H)
{
    return chunk_plan_header_bytes(N) + split_chunk_bound(N, T) * H * (int64_t)R_BYTES;
}

cudaError_t launch_chunk_fp32_split(const ChunkArgs& a, int64_t chunks, cudaStream_t stream)
{
    int32_t* hdr = static_cast<int32_t*>(a.workspace);
    unsigned char* rec = static_cast<unsigned char*>(a.workspace) + chunk_plan_header_bytes(a.N);
    const int64_t units = chunks * a.H;
    if (units > INT32_MAX || 2 * (int64_t)a.N * a.H > INT32_MAX) return cudaErrorInvalidConfiguration;
    cudaError_t e = launch_chunk_plan(a.cu_seqlens, a.N, a.T, hdr, a.status, stream);
    if (e != cudaSuccess) return e;
    if (units > 0) {
        switch (gate_in(a)) {
            case kGateF32: e = launch_prep_gate<kGateF32>(a, hdr, rec, units, stream); break;
            case kGateBF16: e = launch_prep_gate<kGateBF16>(a, hdr, rec, units, stream); break;
            default: e = launch_prep_gate<kGateG>(a, hdr, rec, units, stream); break;
        }
        if (e != cudaSuccess) return e;
    }
    auto kern = a.out_bf16 ? fp32_scan_kernel<__nv_bfloat16> : fp32_scan_kernel<float>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)F_SMEM);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(2 * (int64_t)a.N * a.H), SCAN_THREADS, F_SMEM, stream>>>(a, hdr, rec);
    return cudaGetLastError();
}

}  // namespace kda
