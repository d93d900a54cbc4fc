// Tensor-core chunked KDA forward (tcgen05, TMEM accumulators), sm_103a.
//
// One CTA (256 threads) per (sequence, head); chunks of 64 tokens in order.
// The state is carried transposed, S^T (V x K = 128 x 128): its FP32 master
// lives in registers (thread (v, half) holds S^T[v][64 half .. 64 half + 63])
// and an FP16 copy in shared memory is the A operand of the next chunk's MMAs.
//
// Per chunk (the chunk solve of "Add opt-in FP32 KDA chunk computation",
// sections Problem and Change, in its WY form), with G the in-chunk prefix of
// the log-decay g and a_t = e^{g_t}:
//   A_kk[i][j] = beta_i sum_c k^_ic k^_jc e^{G_ic - G_jc}   (j < i)
//   A_qk[i][j] =        sum_c q^_ic k^_jc e^{G_ic - G_jc}   (j <= i)
//   T' = (I + A_kk)^-1 diag(beta),  X' = K^ o e^G
//   Delta = T' (V - X' S)          (= U - W S with W = T' X', U = T' V)
//   O = scale [(Q^ o e^G) S + A_qk Delta]
//   S <- Diag(e^{G_last}) S + (K^ o e^{G_last - G})^T Delta
// X' S needs only the state entering the chunk, so its MMA runs beside the
// pair sums; once T' is known a single MMA gives Delta.
//
// Pair sums on tensor cores without overflow.  e^{G_i - G_j} is never formed
// as e^{G_i} e^{-G_j} (in-chunk decays reach e^{-1000}).  The 64 tokens are
// split as a binary tree: at level s (blocks of 2s tokens, midpoint m), every
// pair with j in the lower half and i in the upper half of one block factors as
//   e^{G_i - G_j} = (prod_{t=m}^{i} a_t) (prod_{t=j+1}^{m-1} a_t),
// both factors <= 1.  Each level is then a product of "left" rows
// (k^_i or q^_i times the upper factor) with "right" rows (k^_j times the
// lower factor) over the 128 channels; levels 32/16, 8/4, 2/1 are three
// M=128, N=64, K=128 MMAs.  Every pair i > j belongs to exactly one level.
//
// Operands are FP16 (11-bit significand, as TF32, whose precision the
// intra-chunk products need: BF16 operands there cost ~1.6e-3 of output
// rel-L2 each in an FP64 emulation of this algorithm).  In this problem FP16
// underflow only drops contributions far below the error budget.
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
using namespace chunk_ops;

constexpr int DV = kHeadV;    // 128

// Shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t OFF_ST = 0;          // S^T fp16 K-major [128 v][128 c]            32 KiB
constexpr uint32_t OFF_SQ = 32768;      // q staging [64][128] 16-bit -> V^T -> Y^T = (V - X'S)^T fp16 K-major [128 v][64 j]
constexpr uint32_t OFF_SV = 49152;      // v staging [64][128] 16-bit
constexpr uint32_t OFF_SK = 65536;      // k staging -> pair-sum buffer 2 (A part 0)
constexpr uint32_t OFF_SG = 81920;      // g staging fp32 -> pair-sum buffer 2 (A part 1, B)
constexpr uint32_t OFF_AOP = 114688;    // pair-sum buffer 1: A MN-major 2 x 16 KiB, B MN-major 16 KiB
constexpr uint32_t AOP_B = OFF_AOP + 32768;
constexpr uint32_t OFF_AOP2 = OFF_SK;   // pair-sum buffer 2 (after the k and g staging are read)
constexpr uint32_t OFF_AKK = OFF_AOP;                 // after the pair sums: A_kk fp32 [64][68]
constexpr uint32_t OFF_TF = OFF_AOP + C * LDA * 4;    //                      T fp32 [64][68]
constexpr uint32_t OFF_AQK = OFF_AOP + 34816;         //                      A_qk fp16 K-major [64 i][64 j]
constexpr uint32_t OFF_TP = OFF_AOP + 43008;          //                      T' fp16 K-major [64 i][64 j]
constexpr uint32_t OFF_XT = OFF_AOP + 51200;          // X'^T fp16 [128 c][64 j] -> Delta^T K-major [128 v][64 j]
constexpr uint32_t OFF_QP = OFF_XT + 16384;           // Q' fp16 MN-major [128 c][64 i]
constexpr uint32_t OFF_KT = OFF_QP + 16384;           // K''^T fp16 K-major [128 c][64 j]
constexpr uint32_t OFF_RQ = OFF_KT + 16384;           // 1/|q_t|           fp32 [64]
constexpr uint32_t OFF_RK = OFF_RQ + 256;             // 1/|k_t|           fp32 [64]
constexpr uint32_t OFF_DQK = OFF_RK + 256;            // q^_t . k^_t       fp32 [64]
constexpr uint32_t OFF_BETA = OFF_DQK + 256;          // beta              fp32 [64]
constexpr uint32_t OFF_DEC = OFF_BETA + 256;          // e^{G_last}        fp32 [128]
constexpr uint32_t OFF_TOT = OFF_DEC + 512;           // half-chunk decay  fp32 [2][128]
constexpr uint32_t OFF_BAR = OFF_TOT + 1024;          // 6 mbarriers + TMEM slot
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;     // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_TF + C * LDA * 4 <= OFF_AQK && OFF_TP + 8192 <= OFF_XT, "pair-sum region");
static_assert(OFF_AQK % 1024 == 0 && OFF_TP % 1024 == 0 && OFF_XT % 1024 == 0 &&
              OFF_QP % 1024 == 0 && OFF_KT % 1024 == 0 && AOP_B % 1024 == 0 &&
                  OFF_AOP2 + 49152 == OFF_AOP,
              "SW128 tiles need 1024-B alignment");

// TMEM columns.
constexpr uint32_t TM_XS = 0, TM_O = 64, TM_P = 128, TM_A = 256;   // TM_XS: [X'S]^T, then Delta^T
constexpr uint32_t TM_COLS = 512;

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

template <typename TIn, typename TOut, int kGate>
__global__ void __launch_bounds__(NT, 1) chunk_tc_kernel(ChunkArgs args)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    unsigned char* sm = smem_raw + pad;
    const uint32_t sb = raw_s + pad;                      // shared-window address of sm

    float (*akk)[LDA] = reinterpret_cast<float (*)[LDA]>(sm + OFF_AKK);
    float (*Tf)[LDA] = reinterpret_cast<float (*)[LDA]>(sm + OFF_TF);
    const uint16_t* sk = reinterpret_cast<const uint16_t*>(sm + OFF_SK);
    const uint16_t* sq = reinterpret_cast<const uint16_t*>(sm + OFF_SQ);
    const uint16_t* sv = reinterpret_cast<const uint16_t*>(sm + OFF_SV);
    constexpr bool kGated = kGate != kGateG;
    using TG = typename GateSrc<kGate>::T;                 // element of g or f
    constexpr int GP = DK * (int)sizeof(TG) / 16;           // 16-byte pieces per g/f row
    const TG* sg = reinterpret_cast<const TG*>(sm + OFF_SG);
    float* rq = reinterpret_cast<float*>(sm + OFF_RQ);
    float* rk = reinterpret_cast<float*>(sm + OFF_RK);
    float* dqk = reinterpret_cast<float*>(sm + OFF_DQK);
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    float* dec = reinterpret_cast<float*>(sm + OFF_DEC);
    float* tot = reinterpret_cast<float*>(sm + OFF_TOT);
    // [0..2] pair-sum rounds, [3] Delta, [4] output/state update, [5] drain
    // after a failure
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + 56);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane;                     // TMEM lane
    const int ch = tid & 127, hh = tid >> 7;              // channel / token-half ownership
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
    using LD = Loader<TIn>;
    using ST = Stage<TIn>;
    constexpr int P = LD::kPieces;                         // 16-byte pieces per row
    constexpr int NQ = C * P / NT;                         // pieces per thread per tensor
    // 16-bit inputs: the next chunk's loads are issued while this chunk computes.
    constexpr bool kPrefetch = sizeof(TIn) == 2;

    // fused gate: g and beta formed from f, A_log, dt_bias and b (as kda_gate does)
    const TG* __restrict__ graw =
        kGated ? static_cast<const TG*>(args.f) : reinterpret_cast<const TG*>(args.g);
    float lamneg = 0.f, dtb = 0.f;
    if (kGated) {
        lamneg = -expf(args.A_log[h]);
        dtb = args.dt_bias[(int64_t)h * DK + ch];
    }

    // ---- setup: the entering state (zero, or the caller's), TMEM, barriers
    float S[64];                                           // S^T[row][64 half + c]
    if (args.initial_state != nullptr) {
        const float* s0 = args.initial_state + ((int64_t)n * H + h) * DK * DV;
#pragma unroll
        for (int u = 0; u < 64; ++u) S[u] = s0[(int64_t)(64 * half + u) * DV + row];
    } else {
#pragma unroll
        for (int u = 0; u < 64; ++u) S[u] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        uint4 pk;
        pk.x = pack_h2(S[8 * q + 0], S[8 * q + 1]);
        pk.y = pack_h2(S[8 * q + 2], S[8 * q + 3]);
        pk.z = pack_h2(S[8 * q + 4], S[8 * q + 5]);
        pk.w = pack_h2(S[8 * q + 6], S[8 * q + 7]);
        *reinterpret_cast<uint4*>(sm + OFF_ST + sw128_tile(128, row, (64 * half + 8 * q) * 2)) = pk;
    }
    if (warp == 0) {
        tmem_alloc(tslot, TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) mbar_init(&bar[b], 1);
        fence_mbar_init();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tlane = tmem + ((uint32_t)(32 * quad) << 16);

    bool failed = false;
    uint32_t phase = 0;                                    // every barrier completes once per chunk
    // test hook: CTA 0 withholds its first MMA group and the commit that signals it
    const bool withhold = args.fault == KDA_TEST_FAULT_SINGLE_PASS && blockIdx.x == 0;
    // gathers x * 0 over every stored value: NaN once one is infinite or NaN
    float nan_acc = 0.f;

    // 16-bit inputs: each staging region receives the next chunk by cp.async as
    // soon as its last reader in this chunk is done.  FP32 inputs are converted
    // to FP16 on the way in, through registers, at the top of each chunk.
    auto async_rows16 = [&](uint32_t off, const TIn* base, int tc) {
        const int Lc = min(C, eos - tc);
#pragma unroll
        for (int u = 0; u < C * 16 / NT; ++u) {
            const int e = tid + u * NT, r = e >> 4, pc = e & 15;
            const bool ok = r < Lc;
            const TIn* src = base + ((int64_t)(tc + (ok ? r : 0)) * H + h) * DK + pc * 8;
            cp_async16(sm + off + r * 256 + pc * 16, src, ok);
        }
    };
    auto async_g = [&](int tc) {
        const int Lc = min(C, eos - tc);
#pragma unroll
        for (int u = 0; u < C * GP / NT; ++u) {
            const int e = tid + u * NT, r = e / GP, pc = e % GP;
            const bool ok = r < Lc;
            const TG* src = graw + ((int64_t)(tc + (ok ? r : 0)) * H + h) * DK + pc * (16 / (int)sizeof(TG));
            cp_async16(sm + OFF_SG + e * 16, src, ok);
        }
    };
    float xb = 0.f;                                        // beta of this thread's row (tid < 64)
    auto load_beta = [&](int tc) {
        xb = 0.f;
        if (tid < min(C, eos - tc)) {
            const int64_t i = (int64_t)(tc + tid) * H + h;
            if (kGated)
                xb = gate_sigmoid(args.b_bf16
                                      ? __bfloat162float(static_cast<const __nv_bfloat16*>(args.b)[i])
                                      : static_cast<const float*>(args.b)[i]);
            else
                xb = args.beta[i];
        }
    };
    if (kPrefetch && bos < eos) {
        async_rows16(OFF_SQ, gq, bos);
        async_rows16(OFF_SK, gk, bos);
        async_rows16(OFF_SV, gv, bos);
        async_g(bos);
        cp_async_commit();
        load_beta(bos);
    }

    for (int t0 = bos; t0 < eos; t0 += C, phase ^= 1u) {
        const int L = min(C, eos - t0);

        // ---- 1: the chunk in staging (rows >= L zero, decay 1)
        if (kPrefetch) {
            cp_async_wait_all();
        } else {
            // one tensor at a time keeps the FP32 path's registers low
            auto rows_via_regs = [&](const TIn* base, uint32_t off) {
                uint4 x[NQ];
#pragma unroll
                for (int u = 0; u < NQ; ++u) {
                    const int e = tid + u * NT, r = e / P, pc = e % P;
                    x[u] = (r < L) ? LD::load(base + ((int64_t)(t0 + r) * H + h) * DK, pc)
                                   : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < NQ; ++u) {
                    const int e = tid + u * NT, r = e / P, pc = e % P;
                    LD::store(sm + off, r, pc, x[u]);
                }
            };
            rows_via_regs(gq, OFF_SQ);
            rows_via_regs(gk, OFF_SK);
            rows_via_regs(gv, OFF_SV);
            uint4 xg[C * GP / NT];
#pragma unroll
            for (int u = 0; u < C * GP / NT; ++u) {
                const int e = tid + u * NT, r = e / GP, pc = e % GP;
                xg[u] = (r < L) ? __ldg(reinterpret_cast<const uint4*>(
                                      graw + ((int64_t)(t0 + r) * H + h) * DK) + pc)
                                : make_uint4(0, 0, 0, 0);
            }
            load_beta(t0);
#pragma unroll
            for (int u = 0; u < C * GP / NT; ++u) reinterpret_cast<uint4*>(sm + OFF_SG)[tid + u * NT] = xg[u];
        }
        if (tid < C) sbeta[tid] = xb;
        __syncthreads();
        const bool more = kPrefetch && t0 + C < eos;       // a next chunk to prefetch

        // ---- 2: row norms and q^ . k^ (4 threads per row, 32 channels each)
        chunk_norms<TIn>(sm + OFF_SQ, sm + OFF_SK, rq, rk, dqk, args.l2norm != 0, tid);
        __syncthreads();

        // ---- 3: per channel (thread ch, tokens 32 hh .. 32 hh + 31)
        float a[32], kh[32], qh[32];
        {
            // e^g by the hardware exponential, or straight from the gate's input by
            // gate_exp_fast (relative error below 1e-5 either way, far below the FP16
            // operands' rounding); the norms as broadcast 16-byte loads
            const float4* rq4 = reinterpret_cast<const float4*>(rq) + 8 * hh;
            const float4* rk4 = reinterpret_cast<const float4*>(rk) + 8 * hh;
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4) {
                const float4 nq = rq4[u4], nk = rk4[u4];
                const float nqv[4] = {nq.x, nq.y, nq.z, nq.w}, nkv[4] = {nk.x, nk.y, nk.z, nk.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int u = 4 * u4 + e, t = 32 * hh + u;
                    const float gv = load_as_float(sg + t * DK + ch);
                    // rows past the sequence end hold 0: decay 1 in both forms
                    a[u] = kGated ? (t < L ? gate_exp_fast(gv, dtb, lamneg) : 1.f) : __expf(gv);
                    kh[u] = ST::to_f32(sk[t * DK + ch]) * nkv[e];
                    qh[u] = ST::to_f32(sq[t * DK + ch]) * nqv[e];
                }
            }
            float p = 1.f;
#pragma unroll
            for (int u = 0; u < 32; ++u) p *= a[u];
            tot[hh * DK + ch] = p;
        }
        __syncthreads();
        {
            // X'^T = k^ o e^G, Q' = q^ o e^G, K''^T = k^ o e^{G_last - G} (rows of channel ch)
            const float before = hh ? tot[ch] : 1.f;          // decay of tokens before my half
            const float after = hh ? 1.f : tot[DK + ch];      // decay of tokens after my half
            if (hh == 0) dec[ch] = tot[ch] * tot[DK + ch];
            channel_rows(sm + OFF_XT, sm + OFF_QP, sm + OFF_KT, ch, hh, before, after, a, kh, qh);
        }

        // ---- 4: pair sums: three (left x right) MMAs over the channels, the
        // operands of a round written while the previous round's MMA runs
        constexpr uint32_t id_pairs = idesc(kFmtF16, 128, 64, true, true);
        auto issue_round = [&](int rnd, uint32_t buf) {
            fence_async_smem();
            fence_before_sync();
            __syncthreads();
            if (tid == 0 && !(withhold && rnd == 0)) {
                fence_after_sync();
                const uint64_t da = desc_mnmajor128(sb + buf, 16384, 0);
                const uint64_t db = desc_mnmajor64(sb + buf + 32768, 0);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_f16(tmem + TM_A + 64 * rnd, desc_advance(da, mnmajor_off(s)),
                            desc_advance(db, mnmajor_off(s)), id_pairs, s > 0);
                commit(&bar[rnd]);
            }
        };
        auto wait_round = [&](int rnd) -> bool {
            const bool ok = mbar_wait(&bar[rnd], phase);
            return __syncthreads_or(!ok) == 0;
        };
        level32_operands(sm + OFF_AOP, ch, hh, a, kh, qh);
        level_operands<16>(sm + OFF_AOP, ch, hh, 64, 32, a, kh, qh);
        issue_round(0, OFF_AOP);
        if (tid == 0) {
            // [X'S]^T = S^T X'^T and [Q'S]^T = S^T Q'^T need only this chunk's X', Q'
            // and the entering state; the next commit covers them.
            constexpr uint32_t ids = idesc(kFmtF16, 128, 64, false, true);
            const uint64_t dS = desc_kmajor(sb + OFF_ST, 128, 0);
            const uint64_t dX = desc_mnmajor64(sb + OFF_XT, 0), dQ = desc_mnmajor64(sb + OFF_QP, 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_f16(tmem + TM_XS, desc_advance(dS, kmajor_off(128, s)), desc_advance(dX, mnmajor_off(s)), ids,
                        s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_f16(tmem + TM_O, desc_advance(dS, kmajor_off(128, s)), desc_advance(dQ, mnmajor_off(s)), ids,
                        s > 0);
        }
        {
            // V^T fp16 K-major [v][j] into the q staging (q is no longer read)
            float vv[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) vv[u] = ST::to_f32(sv[(32 * hh + u) * DV + ch]);
#pragma unroll
            for (int q = 0; q < 4; ++q) st8(sm + OFF_SQ, 0, ch, 32 * hh + 8 * q, vv + 8 * q);
        }
        level_operands<8>(sm + OFF_AOP2, ch, hh, 0, 0, a, kh, qh);
        level_operands<4>(sm + OFF_AOP2, ch, hh, 64, 32, a, kh, qh);
        issue_round(1, OFF_AOP2);
        if (more) { async_rows16(OFF_SV, gv, t0 + C); cp_async_commit(); }
        if (!wait_round(0)) { failed = true; break; }
        level_operands<2>(sm + OFF_AOP, ch, hh, 0, 0, a, kh, qh);
        level_operands<1>(sm + OFF_AOP, ch, hh, 64, 32, a, kh, qh);
        issue_round(2, OFF_AOP);
        if (!wait_round(1)) { failed = true; break; }
        if (more) {                   // k and g staging (pair-sum buffer 2) are free now
            async_g(t0 + C);
            async_rows16(OFF_SK, gk, t0 + C);
            cp_async_commit();
            load_beta(t0 + C);
        }
        if (!wait_round(2)) { failed = true; break; }
        fence_after_sync();

        // ---- 5: A_kk (fp32) and A_qk (fp16 operand) from TMEM.  The strictly
        // upper part of A_qk is zeroed here, disjoint from the entries written.
        aqk_zero_upper(sm + OFF_AQK, tid);
        extract_pairs(sm + OFF_AQK, &akk[0][0], sbeta, dqk, tlane, TM_A, tid, warp, lane);
        {
            // Y^T[v][j] = V^T[v][j] - [X'S]^T[v][j], in place over the V^T tile
            float xs[32], y[32];
            tmem_ld32(tlane + TM_XS + 32 * half, xs);
            unsigned char* rowp = sm + OFF_SQ;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 pk = *reinterpret_cast<const uint4*>(rowp + sw128(row, (32 * half + 8 * q) * 2));
                const uint32_t w4[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 vf = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
                    y[8 * q + 2 * e] = vf.x - xs[8 * q + 2 * e];
                    y[8 * q + 2 * e + 1] = vf.y - xs[8 * q + 2 * e + 1];
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) st8(rowp, 0, row, 32 * half + 8 * q, y + 8 * q);
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- 6: T = (I + A_kk)^-1: 16x16 diagonal blocks, then the 32- and
        // 64-row merges T_BA = -T_B A_BA T_A.  Y scratch lives in unused upper blocks.
        chunk_inverse(akk, Tf, sbeta, sm + OFF_TP, tid, warp, lane);
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- 7: Delta^T = Y^T T'^T
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t id = idesc(kFmtF16, 128, 64);
            const uint64_t dA = desc_kmajor(sb + OFF_SQ, 128, 0), dT = desc_kmajor(sb + OFF_TP, 64, 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + TM_XS, desc_advance(dA, kmajor_off(128, s)), desc_advance(dT, kmajor_off(64, s)), id,
                        s > 0);
            commit(&bar[3]);
        }
        {
            const bool ok = mbar_wait(&bar[3], phase);
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        if (more) { async_rows16(OFF_SQ, gq, t0 + C); cp_async_commit(); }
        fence_after_sync();
        {
            // Delta^T fp16 K-major [v][i] into the X'^T tile (last read by the X'S MMA)
            float dl[32];
            tmem_ld32(tlane + TM_XS + 32 * half, dl);
#pragma unroll
            for (int q = 0; q < 4; ++q) st8(sm + OFF_XT, 0, row, 32 * half + 8 * q, dl + 8 * q);
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ---- 9: O^T += Delta^T A_qk^T, P^T = Delta^T K''
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t ido = idesc(kFmtF16, 128, 64);
            constexpr uint32_t idp = idesc(kFmtF16, 128, 128);
            const uint64_t dD = desc_kmajor(sb + OFF_XT, 128, 0);
            const uint64_t dAq = desc_kmajor(sb + OFF_AQK, 64, 0), dK = desc_kmajor(sb + OFF_KT, 128, 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + TM_O, desc_advance(dD, kmajor_off(128, s)), desc_advance(dAq, kmajor_off(64, s)), ido,
                        1);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + TM_P, desc_advance(dD, kmajor_off(128, s)), desc_advance(dK, kmajor_off(128, s)), idp,
                        s > 0);
            commit(&bar[4]);
        }
        {
            const bool ok = mbar_wait(&bar[4], phase);
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        fence_after_sync();
        {
            // out = scale O;  S^T <- S^T Diag(d) + P^T;  fp16 copy of S^T
            float o[32];
            tmem_ld32(tlane + TM_O + 32 * half, o);
            const int64_t ostride = (int64_t)H * DV;
            TOut* op = out + ((int64_t)(t0 + 32 * half) * H + h) * DV + row;
            const int nrows = min(32, L - 32 * half);
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                if (u < nrows) {
                    const float y = args.scale * o[u];
                    nan_acc = fmaf(y, 0.f, nan_acc);
                    store_out(op, y);
                }
                op += ostride;
            }
            float p[32];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                tmem_ld32(tlane + TM_P + 64 * half + 32 * part, p);
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    S[32 * part + u] = S[32 * part + u] * dec[64 * half + 32 * part + u] + p[u];
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint4 pk;
                pk.x = pack_h2(S[8 * q + 0], S[8 * q + 1]);
                pk.y = pack_h2(S[8 * q + 2], S[8 * q + 3]);
                pk.z = pack_h2(S[8 * q + 4], S[8 * q + 5]);
                pk.w = pack_h2(S[8 * q + 6], S[8 * q + 7]);
                *reinterpret_cast<uint4*>(sm + OFF_ST + sw128_tile(128, row, (64 * half + 8 * q) * 2)) = pk;
            }
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
    }

    if (kPrefetch) cp_async_wait_all();
    if (failed) {
        if (tid == 0) {
            report_status(args.status, KDA_ERR_TIMEOUT);
            // every MMA this thread issued finishes before the TMEM is released
            commit(&bar[5]);
            mbar_wait(&bar[5], 0);
        }
    } else if (args.final_state != nullptr) {
        float* fs = args.final_state + ((int64_t)n * H + h) * DK * DV;
#pragma unroll
        for (int u = 0; u < 64; ++u) {
            nan_acc = fmaf(S[u], 0.f, nan_acc);
            fs[(int64_t)(64 * half + u) * DV + row] = S[u];
        }
    }
    if (nan_acc != nan_acc) report_status(args.status, KDA_ERR_RANGE);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

template <typename TIn, typename TOut, int kGate>
cudaError_t launch_typed(const ChunkArgs& a, cudaStream_t stream)
{
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel<TIn, TOut, kGate>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.N * a.H;
    if (units > INT32_MAX) return cudaErrorInvalidConfiguration;
    chunk_tc_kernel<TIn, TOut, kGate><<<(unsigned)units, NT, SMEM_BYTES, stream>>>(a);
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

cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t stream)
{
    switch (gate_in(a)) {
        case kGateF32: return launch_gated<kGateF32>(a, stream);
        case kGateBF16: return launch_gated<kGateBF16>(a, stream);
        default: return launch_gated<kGateG>(a, stream);
    }
}

}  // namespace kda
