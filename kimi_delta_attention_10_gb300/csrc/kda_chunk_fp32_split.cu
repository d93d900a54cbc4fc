// FP32-exact chunked KDA forward in two phases, on CUDA cores (IEEE FP32).
//
// The same split as the tensor-core two-phase path ("Add opt-in FP32 KDA chunk
// computation", sections Problem and Change: the chunk solve and the carried
// state, kept in FP32 here):
//   prepare (every (chunk, head) at once, one CTA each):
//     A_kk, A_qk (pair sums with decay factors built from 4- and 16-token
//     sub-blocks, each a product of factors <= 1, so that nothing overflows),
//     T = (I + A_kk)^-1 (16x16 blocks and their merges), W = T X with
//     X = beta k^ o e^G, U = T (beta v), Q' = q^ o e^G,
//     K'' = k^ o e^{G_last - G}, d = e^{G_last}   ->  one FP32 record
//   scan (one CTA per (sequence, head, half of V), chunks in order):
//     Delta = U - W S,  O = scale [Q' S + A_qk Delta],  S <- Diag(d) S + K''^T Delta
// Every product is an FP32 fused multiply-add on CUDA cores, so the mode keeps
// its FP32 accuracy (no TF32 or FP16 operands).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
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

// Record of one unit (FP32, row-major; bytes).
constexpr uint32_t R_W = 0;            // W   [64 i][128 c]
constexpr uint32_t R_QP = 32768;       // Q'  [64 i][128 c]
constexpr uint32_t R_U = 65536;        // U   [64 i][128 v]
constexpr uint32_t R_KT = 98304;       // K'' [64 i][128 c]
constexpr uint32_t R_AQK = 131072;     // A_qk [64 i][64 j] (upper part 0)
constexpr uint32_t R_DEC = 147456;     // d [128]
constexpr uint32_t R_BYTES = 147968;
// the scan brings a record in as two bulk copies: [W, Q', U] and [K'', A_qk, d]
constexpr uint32_t R_EARLY = R_KT, R_LATE = R_BYTES - R_KT;
static_assert(R_BYTES % 16 == 0 && R_EARLY % 16 == 0, "bulk copy sizes");

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
    float* rec = reinterpret_cast<float*>(records + unit * (int64_t)R_BYTES);

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
    // read the same Kb4 rows at once), each lane one row of A_kk or of A_qk
    if (tid < 24 * 8) {
        const int tile = tid >> 3, I = tile / 6, pr = tile % 6;
        const int sa = pr == 0 ? 1 : (pr < 3 ? 2 : 3);      // (sa, sb): (1,0) (2,0) (2,1)
        const int sb = pr == 0 ? 0 : (pr < 3 ? pr - 1 : pr - 3);   //   (3,0) (3,1) (3,2)
        const int i = I * SB + sa * S4 + ((tid >> 1) & 3), rj = I * SB + sb * S4;
        const bool qk = tid & 1;
        const float* x = qk ? &sm.q[i][0] : &sm.k[i][0];
        // sub-blocks strictly between: none, 1, 2 or 1 and 2
        const float* midp = &sm.mid4[I][sa - sb == 1 ? 0 : (sa - sb == 3 ? 3 : sb + 1)][0];
        float acc[S4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c = 0; c < DK; c += 4) {
            const float4 mid = ld4s(midp + c);
            const float4 xv = ld4s(x + c);
#pragma unroll
            for (int u = 0; u < S4; ++u) acc[u] = dot4(xv, mul4(ld4s(&sm.a[rj + u][c]), mid), acc[u]);
        }
        const float s = qk ? 1.f : sm.beta[i];
        st4s(qk ? &sm.aqk[i][rj] : &sm.akk[i][rj],
             make_float4(s * acc[0], s * acc[1], s * acc[2], s * acc[3]));
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
    // lane a 2 x 4 tile of A_kk and of A_qk over all 128 channels (rows r and
    // r + 8: the eight lanes of a quarter warp read eight consecutive rows and
    // one set of Kb16 rows)
    if (tid < 6 * 32) {
        const int pr = tid >> 5, lt = tid & 31;
        const int I = pr == 0 ? 1 : (pr < 3 ? 2 : 3);        // (I, J): (1,0) (2,0) (2,1)
        const int J = pr == 0 ? 0 : (pr < 3 ? pr - 1 : pr - 3);   //   (3,0) (3,1) (3,2)
        const int ib = I * SB + (lt & 7), j0 = J * SB + (lt >> 3) * 4;
        // blocks strictly between: none, 1, 2 or 1 and 2
        const float* midp = &sm.mid16[I - J == 1 ? 0 : (I - J == 3 ? 3 : J + 1)][0];
        float skk[2][4], sqk[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int x = 0; x < 4; ++x) { skk[r][x] = 0.f; sqk[r][x] = 0.f; }
#pragma unroll 2
        for (int c = 0; c < DK; c += 4) {
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
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const float b = sm.beta[ib + 8 * r];
            st4s(&sm.akk[ib + 8 * r][j0],
                 make_float4(b * skk[r][0], b * skk[r][1], b * skk[r][2], b * skk[r][3]));
            st4s(&sm.aqk[ib + 8 * r][j0], make_float4(sqk[r][0], sqk[r][1], sqk[r][2], sqk[r][3]));
        }
    }
    __syncthreads();

    // ---- 7. X = beta k^ o e^G (in place of Kf16), Q' = q^ o e^G and
    // K'' = k^ o e^{G_last - G} to the record, beta v; then A_qk (zero above
    // the diagonal) and d = e^{G_last}
#pragma unroll 2
    for (int m = 0; m < C * DK / 4 / NT; ++m) {
        const int e = tid + NT * m, r = e >> 5, c = (e & 31) * 4, I = r / SB;
        const float4 pre = ld4s(&sm.pre16[I][c]), post = ld4s(&sm.post16[I][c]);
        const float b = sm.beta[r];
        st4s(&sm.k[r][c], scale4(mul4(ld4s(&sm.k[r][c]), pre), b));
        st4s(rec + R_QP / 4 + r * DK + c, mul4(ld4s(&sm.q[r][c]), pre));
        st4s(rec + R_KT / 4 + r * DK + c, mul4(ld4s(&sm.a[r][c]), post));
        st4s(&sm.v[r][c], scale4(ld4s(&sm.v[r][c]), b));
    }
#pragma unroll
    for (int m = 0; m < C * C / 4 / NT; ++m) {
        const int e = tid + NT * m, r = e >> 4, j = (e & 15) * 4;
        const float4 x = ld4s(&sm.aqk[r][j]);
        st4s(rec + R_AQK / 4 + r * C + j, make_float4(j <= r ? x.x : 0.f, j + 1 <= r ? x.y : 0.f,
                                                     j + 2 <= r ? x.z : 0.f, j + 3 <= r ? x.w : 0.f));
    }
    if (tid < DK / 4) {
        const int c = tid * 4;
        st4s(rec + R_DEC / 4 + c, mul4(ld4s(&sm.pre16[NB - 1][c]), ld4s(&sm.blk[NB - 1][c])));
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
        float* dst = rec + (tid < 128 ? R_W : R_U) / 4;
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
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                st4s(dst + (i0 + r) * DK + c0, make_float4(w[r][0], w[r][1], w[r][2], w[r][3]));
                st4s(dst + (i0 + r) * DK + c0 + 4, make_float4(w[r][4], w[r][5], w[r][6], w[r][7]));
            }
        }
    }
}

// ---------------------------------------------------------------- scan
// One CTA per (sequence, head, half of V).  Shared memory holds one record
// (brought in as two bulk copies), the state slice S[c][v] (128 x 64 FP32)
// and Delta (64 x 64).  Per chunk:
//   A: Delta = U - W S and Q S (a 4 x 4 tile of each per thread), then the early
//      part of the next record (W, Q', U) is requested into the freed space;
//   B: O = scale (Q S + A_qk Delta), stored; C: S <- Diag(d) S + K''^T Delta
//      (an 8 x 4 tile per thread); then the late part of the next record.
constexpr int VH = 64;
constexpr int LDS = VH + 4;
constexpr uint32_t F_REC = 0;
constexpr uint32_t F_S = 148480;                        // after the record, 1 KiB aligned
constexpr uint32_t F_D = F_S + DK * LDS * 4;            // Delta [64][68]
constexpr uint32_t F_BAR = F_D + C * LDS * 4;           // 2 mbarriers
constexpr uint32_t F_SMEM = F_BAR + 64;
static_assert(F_S >= R_BYTES && F_SMEM <= 232448, "FP32 scan shared memory");

template <typename TOut>
__global__ void __launch_bounds__(NT, 1) fp32_scan_kernel(ChunkArgs args,
                                                          const int32_t* __restrict__ hdr,
                                                          const unsigned char* __restrict__ records)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char* sm = smem_raw;
    const float* rw = reinterpret_cast<const float*>(sm + F_REC + R_W);
    const float* rq = reinterpret_cast<const float*>(sm + F_REC + R_QP);
    const float* ru = reinterpret_cast<const float*>(sm + F_REC + R_U);
    const float* rk = reinterpret_cast<const float*>(sm + F_REC + R_KT);
    const float* ra = reinterpret_cast<const float*>(sm + F_REC + R_AQK);
    const float* rd = reinterpret_cast<const float*>(sm + F_REC + R_DEC);
    float (*S)[LDS] = reinterpret_cast<float (*)[LDS]>(sm + F_S);
    float (*D)[LDS] = reinterpret_cast<float (*)[LDS]>(sm + F_D);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + F_BAR);   // [0] early part, [1] late part

    const int tid = threadIdx.x;
    const int H = args.H;
    const int vh = blockIdx.x & 1, hb = blockIdx.x >> 1;
    const int n = hdr[kPlanOffsets + args.N + 1 + hb / H], h = hb % H;
    const int bos = args.cu_seqlens[n], eos = args.cu_seqlens[n + 1];
    if (bos < 0 || eos < bos || (int64_t)eos > args.T) return;   // reported by the plan
    const int nch = (eos - bos + C - 1) / C;
    if (hdr[kPlanOffsets + n] + nch > split_chunk_bound(args.N, args.T)) return;   // bad offsets elsewhere
    const int v0 = VH * vh;
    const unsigned char* rec0 =
        records + ((int64_t)hdr[kPlanOffsets + n] * H + h) * (int64_t)R_BYTES;
    const int64_t rstride = (int64_t)H * R_BYTES;
    TOut* __restrict__ out = static_cast<TOut*>(args.out);

    // the entering state slice
    for (int e = tid; e < DK * VH; e += NT) {
        const int c = e / VH, m = e % VH;
        S[c][m] = args.initial_state != nullptr
                      ? args.initial_state[(((int64_t)n * H + h) * DK + c) * DV + v0 + m]
                      : 0.f;
    }
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        if (nch > 0) {
            mbar_arrive_expect_tx(&bar[0], R_EARLY);
            bulk_g2s(sm + F_REC, rec0, R_EARLY, &bar[0]);
            mbar_arrive_expect_tx(&bar[1], R_LATE);
            bulk_g2s(sm + F_REC + R_KT, rec0 + R_KT, R_LATE, &bar[1]);
        }
    }
    __syncthreads();

    // tiles: A and B use rows i0 .. i0 + 3 and columns m0 .. m0 + 3; C uses
    // state rows c0 .. c0 + 7 and columns m0 .. m0 + 3
    const int i0 = (tid >> 4) * 4, m0 = (tid & 15) * 4;
    const int c0 = (tid >> 4) * 8;
    int fail_cc = -1;                                      // chunk whose record did not arrive
    for (int cc = 0; cc < nch; ++cc) {
        const uint32_t par = cc & 1;
        const bool more = cc + 1 < nch;
        const unsigned char* recn = rec0 + (cc + 1) * rstride;
        if (more && tid == 0) bulk_prefetch_l2(recn, R_BYTES);
        {
            const bool ok = mbar_wait(&bar[0], par) && mbar_wait(&bar[1], par);
            if (__syncthreads_or(!ok)) { fail_cc = cc; break; }
        }
        // ---- A: W S and Q' S (K = 128)
        float ws[4][4], qs[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int x = 0; x < 4; ++x) { ws[r][x] = 0.f; qs[r][x] = 0.f; }
        for (int c = 0; c < DK; c += 4) {
            float4 w4[4], q4[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                w4[r] = ld4s(rw + (i0 + r) * DK + c);
                q4[r] = ld4s(rq + (i0 + r) * DK + c);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 s4 = ld4s(&S[c + e][m0]);
                const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const float wv = f4at(w4[r], e), qv = f4at(q4[r], e);
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        ws[r][x] = fmaf(wv, sv[x], ws[r][x]);
                        qs[r][x] = fmaf(qv, sv[x], qs[r][x]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float4 u4 = ld4s(ru + (i0 + r) * DV + v0 + m0);
            *reinterpret_cast<float4*>(&D[i0 + r][m0]) =
                make_float4(u4.x - ws[r][0], u4.y - ws[r][1], u4.z - ws[r][2], u4.w - ws[r][3]);
        }
        __syncthreads();
        // W, Q' and U of this record are read: the next one's early part may come
        if (more && tid == 0) {
            mbar_arrive_expect_tx(&bar[0], R_EARLY);
            bulk_g2s(sm + F_REC, recn, R_EARLY, &bar[0]);
        }
        // ---- B: O = scale (Q' S + A_qk Delta), lower-triangular A_qk
        {
            const int tc = bos + cc * C;
            for (int j = 0; j <= i0 + 3; j += 4) {
                float4 a4[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) a4[r] = ld4s(ra + (i0 + r) * C + j);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 d4 = ld4s(&D[j + e][m0]);
                    const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float av = f4at(a4[r], e);   // 0 above the diagonal
#pragma unroll
                        for (int x = 0; x < 4; ++x) qs[r][x] = fmaf(av, dv[x], qs[r][x]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = tc + i0 + r;
                if (t < eos) {
                    TOut* op = out + ((int64_t)t * H + h) * DV + v0 + m0;
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float y = args.scale * qs[r][x];
                        if constexpr (sizeof(TOut) == 4) op[x] = y;
                        else op[x] = __float2bfloat16_rn(y);
                    }
                }
            }
        }
        // ---- C: S <- Diag(d) S + K''^T Delta (K = 64 tokens)
        {
            float sn[8][4];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float dc = rd[c0 + r];
                const float4 s4 = ld4s(&S[c0 + r][m0]);
                sn[r][0] = dc * s4.x; sn[r][1] = dc * s4.y; sn[r][2] = dc * s4.z; sn[r][3] = dc * s4.w;
            }
            for (int i = 0; i < C; ++i) {
                const float4 ka = ld4s(rk + i * DK + c0), kb = ld4s(rk + i * DK + c0 + 4);
                const float kv[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
                const float4 d4 = ld4s(&D[i][m0]);
                const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int x = 0; x < 4; ++x) sn[r][x] = fmaf(kv[r], dv[x], sn[r][x]);
            }
            __syncthreads();                               // every read of S and the record is done
#pragma unroll
            for (int r = 0; r < 8; ++r)
                *reinterpret_cast<float4*>(&S[c0 + r][m0]) =
                    make_float4(sn[r][0], sn[r][1], sn[r][2], sn[r][3]);
        }
        if (more && tid == 0) {
            mbar_arrive_expect_tx(&bar[1], R_LATE);
            bulk_g2s(sm + F_REC + R_KT, recn + R_KT, R_LATE, &bar[1]);
        }
    }
    __syncthreads();
    if (fail_cc >= 0) {
        // the copies of that chunk's record land (or the wait gives up) before
        // the CTA leaves; no later copy was issued
        if (tid == 0) {
            report_status(args.status, KDA_ERR_TIMEOUT);
            mbar_wait(&bar[0], fail_cc & 1);
            mbar_wait(&bar[1], fail_cc & 1);
        }
        return;
    }
    if (args.final_state != nullptr) {
        for (int e = tid; e < DK * VH; e += NT) {
            const int c = e / VH, m = e % VH;
            args.final_state[(((int64_t)n * H + h) * DK + c) * DV + v0 + m] = S[c][m];
        }
    }
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
    kern<<<(unsigned)(2 * (int64_t)a.N * a.H), NT, F_SMEM, stream>>>(a, hdr, rec);
    return cudaGetLastError();
}

}  // namespace kda
