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
// Every column of S (and of dS) evolves on its own: u, d, dd and du are
// per-column, and only dq^, dk^, dg and dbeta sum over the columns.  So a
// (sequence, head) is split over kSlices CTAs of 32 columns each; each writes
// its partial row sums (slice 0 into the outputs, the others into the
// workspace), and a finishing kernel adds them in slice order and applies the
// norm VJP.
//
// One CTA (256 threads) per (sequence, head, slice) at a time, persistent.
// Lane l of warp w holds rows 4 l.. and slice columns 4 w.. of S and of dS in
// registers (4 x 4): a warp owns whole columns, so the sums over K (u, dd)
// are warp shuffles and a forward token needs no CTA barrier.  The sums over
// the slice's columns (dq^, dk^, dg, dbeta) go through shared memory, one CTA
// barrier per backward token (the buffers of neighbouring tokens alternate).
// Tokens are taken in segments of 16 whose inputs (q^, k^, e^g full rows; v,
// dO slice columns; beta) are staged in shared memory; the raw rows of the
// next segment arrive by cp.async while the current one is processed.
// A first pass stores the state slice at every segment start in the
// workspace; then, segment by segment from the last, the segment is
// recomputed from its checkpoint (the state before each token to a 256 KiB
// per-CTA scratch, u and d to shared memory) and walked backwards, the state
// before the next token loaded while the current one is processed.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <cstddef>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

constexpr int NT = 256;
constexpr int SEG = 16;                                  // tokens per segment
constexpr int DK = kHeadK;
constexpr int DV = kHeadV;
constexpr int kSlices = 4;                               // CTAs per (sequence, head)
constexpr int CW = DV / kSlices;                         // columns per slice
constexpr int64_t kTileBytes = (int64_t)DK * CW * 4;     // one state slice, 16 KiB
constexpr int64_t kTileF4 = kTileBytes / 16;
constexpr int kQ = 4;                                    // float4 per thread per tile
constexpr int kSegPerChunk = kChunk / SEG;               // checkpoint slots per plan chunk
constexpr int kMaxCtas = 1024;                            // persistent CTAs (scratch slots)
constexpr int kCtasPerSm = 2;
static_assert(kQ * 4 * NT == DK * CW, "thread tiles cover the slice");
static_assert(32 * 4 == DK && NT / 32 * 4 == CW, "a lane holds 4 rows, a warp 4 columns");

struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu;
    int32_t N;
    int64_t T;
    int32_t H;
    float scale;
    int32_t l2norm;
    const void* dout;
    const float* init;      // [N,H,K,V] or nullptr
    const float* dfinal;    // [N,H,K,V] or nullptr
    float* dq;              // slice 0's dq^ until the finishing kernel
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    float* dinit;           // or nullptr
    float* part;            // slices 1..: [kSlices-1][3][T,H,K] then [kSlices-1][T,H]
    const int32_t* hdr;     // plan header (chunk offsets)
    float4* ckpt;           // kSegPerChunk * (T/64 + N) * H * kSlices state slices
    float4* scratch;        // gridDim.x * SEG state slices (thread-private float4s)
};

// Shared memory of one CTA (dynamic).
struct BwdSmem {
    float kh[SEG][DK];        // k^ of the segment's tokens
    float qh[SEG][DK];        // q^
    float av[SEG][DK];        // e^g
    float vv[SEG][CW];        // v, dO, d, u: this slice's columns
    float dO[SEG][CW];
    float dl[SEG][CW];
    float uu[SEG][CW];
    float red[2][NT / 32][3][DK];   // per-warp row partials of dq^, dk^, dg (two tokens)
    float dbr[2][NT / 32];          // per-warp partials of dbeta
    float beta[SEG], rq[SEG], rk[SEG];
    // the next segment's raw input rows, brought in by cp.async while the
    // current segment is processed (sized for FP32 inputs)
    unsigned char raw_q[SEG * DK * 4];
    unsigned char raw_k[SEG * DK * 4];
    unsigned char raw_g[SEG * DK * 4];
    unsigned char raw_v[SEG * CW * 4];
    unsigned char raw_do[SEG * CW * 4];
    float raw_beta[SEG];
};

__device__ __forceinline__ float ld1(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ void sst8(float* p, const float (&x)[8])
{
    reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}
// Outputs are written once: streaming stores (__stcs) keep them from
// displacing the state scratch in L2.
// x[lane] for lane < 4 without indexing a register array.
__device__ __forceinline__ float pick4(const float (&x)[4], int lane)
{
    return lane == 0 ? x[0] : lane == 1 ? x[1] : lane == 2 ? x[2] : x[3];
}
__device__ __forceinline__ void f4(const float* p, float* x)
{
    const float4 a = *reinterpret_cast<const float4*>(p);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
}

// 8 (or 4) values of a raw staged row at element c, as float.
__device__ __forceinline__ void raw8(const unsigned char* row, int c, const float*, float (&x)[8])
{
    const float4 a = *reinterpret_cast<const float4*>(row + 4 * c);
    const float4 b = *reinterpret_cast<const float4*>(row + 4 * c + 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void raw8(const unsigned char* row, int c, const __nv_bfloat16*, float (&x)[8])
{
    const uint4 u = *reinterpret_cast<const uint4*>(row + 2 * c);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}
__device__ __forceinline__ float4 raw4(const unsigned char* row, int c, const float*)
{
    return *reinterpret_cast<const float4*>(row + 4 * c);
}
__device__ __forceinline__ float4 raw4(const unsigned char* row, int c, const __nv_bfloat16*)
{
    const uint2 u = *reinterpret_cast<const uint2*>(row + 2 * c);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src)
                 : "memory");
}

// Sum over the warp's 32 lanes (K rows) of p[j], j < 4 (the warp's columns):
// every lane returns all four sums.  A transpose-reduction (lanes 16 apart
// split the columns in halves, lanes 8 apart in quarters, then a butterfly
// over the remaining 8 lanes) leaves column 2 b4 + b3 in the lanes with
// bits (b4, b3); four shuffles broadcast them.
__device__ __forceinline__ void ksum_warp(const float (&p)[4], int lane, float (&out)[4])
{
    const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1;
    float q2[2];
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const float keep = b4 ? p[2 + m] : p[m], send = b4 ? p[m] : p[2 + m];
        q2[m] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float q1 = (b3 ? q2[1] : q2[0]) + __shfl_xor_sync(0xffffffffu, b3 ? q2[0] : q2[1], 8);
    q1 += __shfl_xor_sync(0xffffffffu, q1, 4);
    q1 += __shfl_xor_sync(0xffffffffu, q1, 2);
    q1 += __shfl_xor_sync(0xffffffffu, q1, 1);
#pragma unroll
    for (int j = 0; j < 4; ++j) out[j] = __shfl_sync(0xffffffffu, q1, 8 * j);
}

template <typename TIn, typename TO>
__global__ void __launch_bounds__(NT, kCtasPerSm) chunk_bwd_kernel(BwdArgs a)
{
    extern __shared__ float4 dyn_smem[];
    BwdSmem& sm = *reinterpret_cast<BwdSmem*>(dyn_smem);

    // lane = row group (rows 4 lane ..), warp = column group (slice columns 4 warp ..)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H;
    const TIn* gq = static_cast<const TIn*>(a.q);
    const TIn* gk = static_cast<const TIn*>(a.k);
    const TIn* gv = static_cast<const TIn*>(a.v);
    const TO* gdo = static_cast<const TO*>(a.dout);
    float4* scratch = a.scratch + (int64_t)blockIdx.x * SEG * kTileF4;
    const int64_t THK = a.T * H * DK, TH = a.T * H;
    const int tofs = warp * kQ * 32 + lane;                // this thread's float4 q of a tile: tofs + 32 q
    int tok = 0;                                           // parity of the row-sum buffers

    const int64_t units = (int64_t)a.N * H * kSlices;
    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
        const int vs = (int)(unit % kSlices);
        const int64_t nh = unit / kSlices;                 // n * H + h
        const int n = (int)(nh / H), h = (int)(nh % H);
        const int c0 = CW * vs;                            // first column of the slice
        const int cw = 4 * warp;                           // the warp's first column in the slice
        const int bos = a.cu[n], eos = a.cu[n + 1];
        if (bos < 0 || eos < bos || (int64_t)eos > a.T) continue;   // reported by the plan
        const int nseg = (eos - bos + SEG - 1) / SEG;
        float4* ck = a.ckpt +
                     (((int64_t)kSegPerChunk * a.hdr[kPlanOffsets + n] * H + h) * kSlices + vs) * kTileF4;
        const int64_t ck_stride = (int64_t)H * kSlices * kTileF4;
        float* pq = vs == 0 ? a.dq : a.part + ((int64_t)(vs - 1) * 3 + 0) * THK;
        float* pk = vs == 0 ? a.dk : a.part + ((int64_t)(vs - 1) * 3 + 1) * THK;
        float* pg = vs == 0 ? a.dg : a.part + ((int64_t)(vs - 1) * 3 + 2) * THK;
        float* pb = vs == 0 ? a.dbeta : a.part + (int64_t)(kSlices - 1) * 3 * THK + (vs - 1) * TH;

        // The segment's raw input rows (k, g, v, beta and, with_bwd, q and dO)
        // into the raw buffers by cp.async; rows >= L are not loaded.
        auto issue = [&](int t0, int L, bool with_bwd) {
            constexpr int kRow = DK * (int)sizeof(TIn), kCpr = kRow / 16;     // q, k rows
            constexpr int vRow = CW * (int)sizeof(TIn), vCpr = vRow / 16;     // v slice rows
            constexpr int oRow = CW * (int)sizeof(TO), oCpr = oRow / 16;      // dO slice rows
            for (int e = tid; e < SEG * kCpr; e += NT) {
                const int r = e / kCpr, pc = e % kCpr;
                if (r < L) {
                    const int64_t row = ((int64_t)(t0 + r) * H + h) * DK;
                    tc::cp_async16(sm.raw_k + r * kRow + 16 * pc,
                                   reinterpret_cast<const unsigned char*>(gk + row) + 16 * pc, true);
                    if (with_bwd)
                        tc::cp_async16(sm.raw_q + r * kRow + 16 * pc,
                                       reinterpret_cast<const unsigned char*>(gq + row) + 16 * pc, true);
                }
            }
            for (int e = tid; e < SEG * 32; e += NT) {                           // g: 512-byte rows
                const int r = e >> 5, pc = e & 31;
                if (r < L)
                    tc::cp_async16(sm.raw_g + r * 512 + 16 * pc,
                                   a.g + ((int64_t)(t0 + r) * H + h) * DK + 4 * pc, true);
            }
            for (int e = tid; e < SEG * vCpr; e += NT) {
                const int r = e / vCpr, pc = e % vCpr;
                if (r < L)
                    tc::cp_async16(sm.raw_v + r * vRow + 16 * pc,
                                   reinterpret_cast<const unsigned char*>(
                                       gv + ((int64_t)(t0 + r) * H + h) * DV + c0) + 16 * pc, true);
            }
            if (with_bwd) {
                for (int e = tid; e < SEG * oCpr; e += NT) {
                    const int r = e / oCpr, pc = e % oCpr;
                    if (r < L)
                        tc::cp_async16(sm.raw_do + r * oRow + 16 * pc,
                                       reinterpret_cast<const unsigned char*>(
                                           gdo + ((int64_t)(t0 + r) * H + h) * DV + c0) + 16 * pc, true);
                }
            }
            if (tid < L) cp_async4(&sm.raw_beta[tid], a.beta + (int64_t)(t0 + tid) * H + h);
            tc::cp_async_commit();
        };
        // The issued segment in the working arrays: q^, k^ (normalised rows),
        // e^g, the slice of v and (with_bwd) dO, beta; rows >= L unused.
        auto finish = [&](int L, bool with_bwd) {
            tc::cp_async_wait_all();
            __syncthreads();                               // the raw rows landed; the previous segment is done
            {
                const int r = tid >> 4, c = 8 * (tid & 15);
                if (r < L) {
                    float x[8];
                    raw8(sm.raw_k + r * DK * (int)sizeof(TIn), c, gk, x);
                    sst8(&sm.kh[r][c], x);
                    raw8(sm.raw_g + r * DK * 4, c, a.g, x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = expf(x[e]);
                    sst8(&sm.av[r][c], x);
                    if (with_bwd) {
                        raw8(sm.raw_q + r * DK * (int)sizeof(TIn), c, gq, x);
                        sst8(&sm.qh[r][c], x);
                    }
                }
            }
            if (tid < SEG * CW / 4) {
                const int r = tid >> 3, c = 4 * (tid & 7);
                if (r < L) {
                    *reinterpret_cast<float4*>(&sm.vv[r][c]) = raw4(sm.raw_v + r * CW * (int)sizeof(TIn), c, gv);
                    if (with_bwd)
                        *reinterpret_cast<float4*>(&sm.dO[r][c]) = raw4(sm.raw_do + r * CW * (int)sizeof(TO), c, gdo);
                }
            }
            if (tid < SEG) sm.beta[tid] = tid < L ? sm.raw_beta[tid] : 0.f;
            __syncthreads();
            // row norms: warp w takes rows 2 w and 2 w + 1
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int r = 2 * warp + rr;
                if (r < L) {
                    float sk = 0.f, sq = 0.f, x4[4];
                    f4(&sm.kh[r][4 * lane], x4);
#pragma unroll
                    for (int e = 0; e < 4; ++e) sk += x4[e] * x4[e];
                    if (with_bwd) {
                        f4(&sm.qh[r][4 * lane], x4);
#pragma unroll
                        for (int e = 0; e < 4; ++e) sq += x4[e] * x4[e];
                    }
#pragma unroll
                    for (int m = 16; m > 0; m >>= 1) {
                        sk += __shfl_xor_sync(0xffffffffu, sk, m);
                        sq += __shfl_xor_sync(0xffffffffu, sq, m);
                    }
                    if (lane == 0) {
                        sm.rk[r] = a.l2norm ? 1.f / sqrtf(sk + 1e-6f) : 1.f;
                        sm.rq[r] = a.l2norm ? 1.f / sqrtf(sq + 1e-6f) : 1.f;
                    }
                }
            }
            __syncthreads();
            {
                const int r = tid >> 4, c = 8 * (tid & 15);
                if (r < L) {
                    float x[8];
                    const float nk = sm.rk[r], nq = sm.rq[r];
                    f4(&sm.kh[r][c], x);
                    f4(&sm.kh[r][c + 4], x + 4);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] *= nk;
                    sst8(&sm.kh[r][c], x);
                    if (with_bwd) {
                        f4(&sm.qh[r][c], x);
                        f4(&sm.qh[r][c + 4], x + 4);
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] *= nq;
                        sst8(&sm.qh[r][c], x);
                    }
                }
            }
            __syncthreads();                               // working arrays ready; raw buffers free
        };
        // One forward token: S <- S' + k^ d^T with S' = Diag(a) S; u and d of
        // the token to uu / dl row tl when `keep`.  Warp-local: no barrier.
        auto fwd_token = [&](float (&S)[16], int tl, bool keep) {
            float av4[4], kn[4], p[4], u[4], vv4[4];
            f4(&sm.av[tl][4 * lane], av4);
            f4(&sm.kh[tl][4 * lane], kn);
            f4(&sm.vv[tl][cw], vv4);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) S[4 * i + j] *= av4[i];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) acc += S[4 * i + j] * kn[i];
                p[j] = acc;
            }
            ksum_warp(p, lane, u);
            const float bt = sm.beta[tl];
            float d4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) d4[j] = bt * (vv4[j] - u[j]);
            if (keep && lane < 4) {
                sm.uu[tl][cw + lane] = pick4(u, lane);
                sm.dl[tl][cw + lane] = pick4(d4, lane);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) S[4 * i + j] += kn[i] * d4[j];
        };
        // This thread's 4 x 4 block of a caller state [N,H,K,V] (zero if none).
        auto load_state = [&](const float* src, float (&S)[16]) {
            if (src == nullptr) {
#pragma unroll
                for (int e = 0; e < 16; ++e) S[e] = 0.f;
                return;
            }
            const float* s0 = src + nh * DK * DV;
#pragma unroll
            for (int i = 0; i < 4; ++i) f4(s0 + (4 * lane + i) * DV + c0 + cw, S + 4 * i);
        };
        auto tstore = [&](float4* base, const float (&s)[16]) {
#pragma unroll
            for (int q = 0; q < kQ; ++q)
                base[tofs + 32 * q] = make_float4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]);
        };
        auto tload = [&](const float4* base, float (&s)[16]) {
#pragma unroll
            for (int q = 0; q < kQ; ++q) {
                const float4 x = base[tofs + 32 * q];
                s[4 * q] = x.x; s[4 * q + 1] = x.y; s[4 * q + 2] = x.z; s[4 * q + 3] = x.w;
            }
        };

        // ---- forward pass: the state slice at every segment start
        float S[16];
        load_state(a.init, S);
        auto seg_len = [&](int sg) { return min(SEG, eos - (bos + sg * SEG)); };
        if (nseg > 0) issue(bos, seg_len(0), false);
        for (int sg = 0; sg < nseg; ++sg) {
            const int L = seg_len(sg);
            tstore(ck + sg * ck_stride, S);
            finish(L, false);
            if (sg + 1 < nseg) issue(bos + (sg + 1) * SEG, seg_len(sg + 1), false);
            for (int tl = 0; tl < L; ++tl) fwd_token(S, tl, false);
        }

        // ---- backward, segment by segment from the last
        float dS[16];
        load_state(a.dfinal, dS);
        if (nseg > 0) issue(bos + (nseg - 1) * SEG, seg_len(nseg - 1), true);
        for (int sg = nseg - 1; sg >= 0; --sg) {
            const int t0 = bos + sg * SEG, L = seg_len(sg);
            // recompute the segment: the state before each token, u and d
            tload(ck + sg * ck_stride, S);
            finish(L, true);
            if (sg > 0) issue(bos + (sg - 1) * SEG, seg_len(sg - 1), true);
            for (int tl = 0; tl < L; ++tl) {
                tstore(scratch + (int64_t)tl * kTileF4, S);
                fwd_token(S, tl, true);
            }
            __syncthreads();                               // u and d of every column in place
            // walk it backwards; the state before token tl - 1 is loaded while
            // token tl is processed (each thread reads back what it wrote)
            float Snext[16];
            tload(scratch + (int64_t)(L - 1) * kTileF4, Snext);
            for (int tl = L - 1; tl >= 0; --tl) {
                const int64_t t = t0 + tl;
                float Sp[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) Sp[e] = Snext[e];
                if (tl > 0) tload(scratch + (int64_t)(tl - 1) * kTileF4, Snext);
                float av4[4], kn[4], qn[4], dO[4], d4[4], vv4[4], uu4[4];
                f4(&sm.av[tl][4 * lane], av4);
                f4(&sm.kh[tl][4 * lane], kn);
                f4(&sm.qh[tl][4 * lane], qn);
                f4(&sm.dO[tl][cw], dO);
                f4(&sm.dl[tl][cw], d4);
                f4(&sm.vv[tl][cw], vv4);
                f4(&sm.uu[tl][cw], uu4);
                const float bt = sm.beta[tl];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) Sp[4 * i + j] *= av4[i];
                // o = scale S^T q^:  dS += scale q^ dO^T,  dq^ = scale S dO
                float dqn[4], ddp[4], dd[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc += (Sp[4 * i + j] + kn[i] * d4[j]) * dO[j];
                        dS[4 * i + j] += a.scale * qn[i] * dO[j];
                    }
                    dqn[i] = a.scale * acc;
                }
                // dd = dS^T k^ (over all K rows: the warp)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc += dS[4 * i + j] * kn[i];
                    ddp[j] = acc;
                }
                ksum_warp(ddp, lane, dd);
                float du[4], dbw = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    du[j] = -bt * dd[j];
                    dbw += dd[j] * (vv4[j] - uu4[j]);
                }
                if (lane < 4) __stcs(&a.dv[(t * H + h) * DV + c0 + cw + lane], bt * pick4(dd, lane));
                // dk^ = dS d + S' du;  dS' = dS + k^ du^T;  dg = rowsum(dS' o S');  dS = a dS'
                float dkn[4], dgp[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float acc = 0.f, accg = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc += dS[4 * i + j] * d4[j] + Sp[4 * i + j] * du[j];
                        const float dsp = dS[4 * i + j] + kn[i] * du[j];
                        accg += dsp * Sp[4 * i + j];
                        dS[4 * i + j] = av4[i] * dsp;
                    }
                    dkn[i] = acc;
                    dgp[i] = accg;
                }
                // the warp's row partials (its 4 columns) to shared memory; the
                // sums over the slice's 8 warps after one barrier
                const int buf = tok++ & 1;
                *reinterpret_cast<float4*>(&sm.red[buf][warp][0][4 * lane]) = make_float4(dqn[0], dqn[1], dqn[2], dqn[3]);
                *reinterpret_cast<float4*>(&sm.red[buf][warp][1][4 * lane]) = make_float4(dkn[0], dkn[1], dkn[2], dkn[3]);
                *reinterpret_cast<float4*>(&sm.red[buf][warp][2][4 * lane]) = make_float4(dgp[0], dgp[1], dgp[2], dgp[3]);
                if (lane == 0) sm.dbr[buf][warp] = dbw;
                __syncthreads();
                for (int o = tid; o < 3 * DK; o += NT) {
                    const int qv = o / DK, r = o % DK;
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < NT / 32; ++w) acc += sm.red[buf][w][qv][r];
                    float* dst = qv == 0 ? pq : (qv == 1 ? pk : pg);
                    __stcs(&dst[(t * H + h) * DK + r], acc);
                }
                if (tid == 0) {
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < NT / 32; ++w) acc += sm.dbr[buf][w];
                    pb[t * H + h] = acc;
                }
            }
        }
        if (a.dinit != nullptr) {
            float* d0 = a.dinit + nh * DK * DV;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(d0 + (4 * lane + i) * DV + c0 + cw) =
                    make_float4(dS[4 * i], dS[4 * i + 1], dS[4 * i + 2], dS[4 * i + 3]);
        }
    }
}

// The slices' partial row sums added in slice order (slice 0 already in the
// outputs), then the norm VJP dx = (dx^ - x^ (x^ . dx^)) / n with
// n = sqrt(|x|^2 + eps) for q and k when l2norm; one warp per (token, head) row.
template <typename TIn>
__global__ void __launch_bounds__(256) bwd_finish_kernel(const TIn* __restrict__ q,
                                                         const TIn* __restrict__ k,
                                                         float* __restrict__ dq,
                                                         float* __restrict__ dk,
                                                         float* __restrict__ dg,
                                                         float* __restrict__ dbeta,
                                                         const float* __restrict__ part,
                                                         int64_t rows, int32_t l2norm)
{
    const int lane = threadIdx.x & 31;
    const int64_t THK = rows * DK;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nw) {
        const int64_t o = r * DK + 4 * lane;
        float4 sq = *reinterpret_cast<const float4*>(dq + o);
        float4 sk = *reinterpret_cast<const float4*>(dk + o);
        float4 sg = *reinterpret_cast<const float4*>(dg + o);
#pragma unroll
        for (int s = 1; s < kSlices; ++s) {
            const float* base = part + (int64_t)(s - 1) * 3 * THK;
            const float4 pq = *reinterpret_cast<const float4*>(base + o);
            const float4 pk = *reinterpret_cast<const float4*>(base + THK + o);
            const float4 pg = *reinterpret_cast<const float4*>(base + 2 * THK + o);
            sq.x += pq.x; sq.y += pq.y; sq.z += pq.z; sq.w += pq.w;
            sk.x += pk.x; sk.y += pk.y; sk.z += pk.z; sk.w += pk.w;
            sg.x += pg.x; sg.y += pg.y; sg.z += pg.z; sg.w += pg.w;
        }
        *reinterpret_cast<float4*>(dg + o) = sg;
        if (lane == 0) {
            float b = dbeta[r];
            for (int s = 1; s < kSlices; ++s) b += part[(int64_t)(kSlices - 1) * 3 * THK + (s - 1) * rows + r];
            dbeta[r] = b;
        }
        auto norm_vjp = [&](const TIn* x, float4 gv4, float* out) {
            if (!l2norm) {
                *reinterpret_cast<float4*>(out + o) = gv4;
                return;
            }
            const float gv[4] = {gv4.x, gv4.y, gv4.z, gv4.w};
            float xv[4], ss = 0.f, dot = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                xv[e] = ld1(x, o + e);
                ss += xv[e] * xv[e];
                dot += xv[e] * gv[e];
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                ss += __shfl_xor_sync(0xffffffffu, ss, m);
                dot += __shfl_xor_sync(0xffffffffu, dot, m);
            }
            const float inv = 1.f / sqrtf(ss + 1e-6f);
            const float proj = dot * inv * inv;             // (x^ . dx^) / n
            *reinterpret_cast<float4*>(out + o) =
                make_float4((gv[0] - xv[0] * proj) * inv, (gv[1] - xv[1] * proj) * inv,
                            (gv[2] - xv[2] * proj) * inv, (gv[3] - xv[3] * proj) * inv);
        };
        norm_vjp(q, sq, dq);
        norm_vjp(k, sk, dk);
    }
}

template <typename TIn, typename TO>
cudaError_t launch_typed(const BwdArgs& a, int grid, cudaStream_t stream)
{
    constexpr int smem = (int)sizeof(BwdSmem);
    cudaError_t e = cudaFuncSetAttribute(chunk_bwd_kernel<TIn, TO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_bwd_kernel<TIn, TO><<<grid, NT, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.T == 0) return e;
    const int64_t rows = a.T * a.H;
    const int sms = device_sm_count();
    const int64_t blocks = std::min<int64_t>((rows + 7) / 8, (int64_t)(sms > 0 ? sms : 152) * 8);
    bwd_finish_kernel<TIn><<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), a.dq, a.dk, a.dg, a.dbeta,
        a.part, rows, a.l2norm);
    return cudaGetLastError();
}

int64_t ckpt_bytes(int32_t N, int64_t T, int32_t H)
{
    return kSegPerChunk * split_chunk_bound(N, T) * H * kSlices * kTileBytes;
}
int64_t part_bytes(int64_t T, int32_t H)
{
    return (int64_t)(kSlices - 1) * (3 * T * H * DK + T * H) * 4;
}
int64_t bwd_ctas(int32_t N, int32_t H)
{
    const int sms = device_sm_count();
    return std::min<int64_t>((int64_t)N * H * kSlices,
                             std::min<int64_t>(kMaxCtas, (int64_t)kCtasPerSm * (sms > 0 ? sms : 152)));
}

}  // namespace

int64_t bwd_workspace_bytes(int32_t N, int64_t T, int32_t H)
{
    // the scratch is sized for the CTA cap, not this device's SM count
    const int64_t ctas = std::min<int64_t>((int64_t)N * H * kSlices, kMaxCtas);
    const int64_t part = (part_bytes(T, H) + 255) / 256 * 256;
    return chunk_plan_header_bytes(N) + ckpt_bytes(N, T, H) + part + ctas * SEG * kTileBytes;
}

cudaError_t launch_chunk_bwd(const BwdLaunch& L, cudaStream_t stream)
{
    static_assert(sizeof(BwdSmem) * kCtasPerSm <= 227 * 1024, "shared memory budget");
    static_assert(offsetof(BwdSmem, red) % 16 == 0, "16-byte shared stores");
    const int64_t units = (int64_t)L.N * L.H * kSlices;
    const int grid = (int)bwd_ctas(L.N, L.H);
    int32_t* hdr = static_cast<int32_t*>(L.workspace);
    unsigned char* ws = static_cast<unsigned char*>(L.workspace) + chunk_plan_header_bytes(L.N);
    BwdArgs a;
    a.q = L.q; a.k = L.k; a.v = L.v; a.g = L.g; a.beta = L.beta;
    a.cu = L.cu; a.N = L.N; a.T = L.T; a.H = L.H; a.scale = L.scale; a.l2norm = L.l2norm;
    a.dout = L.dout; a.init = L.init; a.dfinal = L.dfinal;
    a.dq = L.dq; a.dk = L.dk; a.dv = L.dv; a.dg = L.dg; a.dbeta = L.dbeta; a.dinit = L.dinit;
    a.hdr = hdr;
    a.ckpt = reinterpret_cast<float4*>(ws);
    ws += ckpt_bytes(L.N, L.T, L.H);
    a.part = reinterpret_cast<float*>(ws);
    ws += (part_bytes(L.T, L.H) + 255) / 256 * 256;
    a.scratch = reinterpret_cast<float4*>(ws);
    cudaError_t e = launch_chunk_plan(L.cu, L.N, L.T, hdr, L.status, stream);
    if (e != cudaSuccess || units == 0) return e;
    if (L.qkv_bf16)
        return L.dout_bf16 ? launch_typed<__nv_bfloat16, __nv_bfloat16>(a, grid, stream)
                           : launch_typed<__nv_bfloat16, float>(a, grid, stream);
    return L.dout_bf16 ? launch_typed<float, __nv_bfloat16>(a, grid, stream)
                       : launch_typed<float, float>(a, grid, stream);
}

}  // namespace kda
