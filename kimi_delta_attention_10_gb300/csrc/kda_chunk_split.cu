// Two-phase tensor-core chunked KDA forward (tcgen05, TMEM accumulators), sm_103a.
//
// The chunk solve ("Add opt-in FP32 KDA chunk computation", sections Problem
// and Change, in its WY form) splits into a part that needs only the chunk's
// own inputs and a short part that needs the state entering the chunk:
//   prepare:  A_kk, A_qk (pair sums), T' = (I + A_kk)^-1 diag(beta),
//             W = T' (K^ o e^G),  U = T' V,  Q' = Q^ o e^G,
//             K'' = K^ o e^{G_last - G},  d = e^{G_last}
//   scan:     Delta = U - W S
//             O = scale [Q' S + A_qk Delta]
//             S <- Diag(d) S + K''^T Delta
// The preparation of every (chunk, head) is independent, so it runs over the
// whole problem at once on every SM (chunk_prep_kernel: one CTA per unit, two
// CTAs per SM); its results go to a caller-provided workspace as one record
// per unit, already in the 128-byte-swizzled layouts the scan's MMAs read.
// The scan (chunk_scan_kernel: one CTA per (sequence, head)) then walks the
// chunks in order with the state on chip, bringing each record in by one bulk
// copy, double-buffered, while it works on the one before.  A plan kernel
// first turns cu_seqlens into per-sequence chunk offsets.  When the scan CTAs
// alone would leave SMs idle, the chunks are cut into windows so that the
// preparation of later chunks runs beside the scan of earlier ones (see
// launch_chunk_split).
//
// Record of one unit (bytes), in this order:
//   W       fp16 [128 c][64 i]  (MN-major B of [W S]^T = S^T W^T)
//   Q'      fp16 [128 c][64 i]  (MN-major B of [Q' S]^T)
//   U^T     fp16 [128 v][64 i]  (row v read by the thread of state row v)
//   A_qk    fp16 [64 i][64 j]   (K-major B of [A_qk Delta]^T; strictly upper part 0)
//   K''^T   fp16 [128 c][64 j]  (K-major B of [K''^T Delta]^T)
//   d       fp32 [128]
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "kda_internal.cuh"
#include "kda_tc.cuh"
#include "kda_chunk_ops.cuh"

namespace kda {

namespace {

using namespace tc;
using namespace chunk_ops;

constexpr int DV = kHeadV;

constexpr uint32_t REC_W = 0;
constexpr uint32_t REC_QP = 16384;
constexpr uint32_t REC_U = 32768;
constexpr uint32_t REC_AQK = 49152;
constexpr uint32_t REC_KT = 57344;
constexpr uint32_t REC_DEC = 73728;
constexpr uint32_t REC_BYTES = 74240;
static_assert(REC_BYTES % 16 == 0 && REC_BYTES < (1u << 20), "bulk copy size");

// Workspace header: int32 [0] = 1 when the plan found offsets outside [0, T]
// or out of order (those sequences get no chunks and are skipped; the chunks
// of the others can then add up past the T / 64 + N records the workspace
// holds, and the scans skip every sequence whose records would lie past
// that bound), int32 [4 .. 4 + N] = chunk
// offsets (chunks of sequences 0 .. n-1), then int32 [5 + N .. 5 + 2N) = the
// order in which the scan takes the sequences: longest first (LPT), so that
// short sequences fill the tail of a packed batch (input order above
// kLptMaxSeqs sequences), then int32 [5 + 2N .. 5 + 2N + kMaxWindows) = the
// unit counters the preparation CTAs of each chunk window take work from
// (zeroed by the plan).
constexpr int kHdrOff = 4;
constexpr int kLptMaxSeqs = 1024;
constexpr int kMaxWindows = 3;

int64_t header_bytes(int32_t N)
{
    return ((int64_t)(kHdrOff + 2 * N + 1 + kMaxWindows) * 4 + 1023) / 1024 * 1024;
}
__host__ __device__ int32_t* window_counters(int32_t* hdr, int32_t N) { return hdr + kHdrOff + 2 * N + 1; }

// ---------------------------------------------------------------- plan
__global__ void __launch_bounds__(1024) chunk_plan_kernel(const int32_t* __restrict__ cu, int32_t N,
                                                          int64_t T, int32_t* __restrict__ hdr,
                                                          int32_t* status)
{
    __shared__ int32_t wsum[32];
    __shared__ int32_t carry;
    __shared__ int32_t bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t* off = hdr + kHdrOff;
    if (tid == 0) {
        carry = 0;
        bad = 0;
        off[0] = 0;
    }
    __syncthreads();
    for (int32_t base = 0; base < N; base += 1024) {
        const int32_t n = base + tid;
        int32_t cnt = 0;
        if (n < N) {
            const int32_t bos = cu[n], eos = cu[n + 1];
            if (bos < 0 || eos < bos || (int64_t)eos > T) bad = 1;   // no chunks: skipped
            else cnt = (eos - bos + kChunk - 1) / kChunk;
        }
        int32_t x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int32_t incl = carry + x + (warp > 0 ? wsum[warp - 1] : 0);
        if (n < N) off[n + 1] = incl;
        __syncthreads();
        if (tid == 1023) carry = incl;
        __syncthreads();
    }
    if (tid == 0) {
        hdr[0] = bad;
        if (bad) report_status(status, KDA_ERR_DEVICE_ARG);
    }
    if (tid < kMaxWindows) window_counters(hdr, N)[tid] = 0;
    // scan order: rank of each sequence by length, longest first, ties by index
    int32_t* order = hdr + kHdrOff + N + 1;
    if (N <= kLptMaxSeqs) {
        __shared__ int32_t len[kLptMaxSeqs];
        if (tid < N) {
            const int32_t bos = cu[tid], eos = cu[tid + 1];
            len[tid] = (bos < 0 || eos < bos || (int64_t)eos > T) ? 0 : eos - bos;
        }
        __syncthreads();
        if (tid < N) {
            const int32_t mine = len[tid];
            int32_t rank = 0;
            for (int32_t m = 0; m < N; ++m) {
                const int32_t other = len[m];
                rank += (other > mine) || (other == mine && m < tid);
            }
            order[rank] = tid;
        }
    } else {
        for (int32_t n = tid; n < N; n += 1024) order[n] = n;
    }
}

// ---------------------------------------------------------------- prepare
// Shared memory of one preparation CTA (bytes from a 1024-aligned base).  The
// staging of q, k and g is dead once every thread holds its channel's values
// in registers; the pair-sum operands, X'^T and then A_kk / T reuse it.
constexpr uint32_t P_SQ = 0;           // q staging [64][128] 16-bit
constexpr uint32_t P_SK = 16384;       // k staging
constexpr uint32_t P_SG = 32768;       // g (or f) staging fp32 [64][128]
constexpr uint32_t P_PAIR = 0;         // pair-sum operands: A MN-major 2 x 16 KiB, B 16 KiB
constexpr uint32_t P_AKK = 0;          // after the pair sums: A_kk fp32 [64][68]
constexpr uint32_t P_TF = C * LDA * 4; //                      T fp32 [64][68]
constexpr uint32_t P_XT = 49152;       // X'^T fp16 K-major [128 c][64 j]
constexpr uint32_t P_SV = 65536;       // v staging -> V^T fp16 K-major [128 v][64 j]
constexpr uint32_t P_AQK = 81920;      // A_qk fp16 [64 i][64 j]
constexpr uint32_t P_TP = 90112;       // T' fp16 [64 i][64 j]
// Until T' is written (the end of the inverse) its region holds the unit's
// small vectors: beta (read into registers before the inverse's last
// barrier), the norms, q^.k^ and the half-chunk decay products.
constexpr uint32_t P_BETA = P_TP;          // beta fp32 [64]
constexpr uint32_t P_RQ = P_TP + 256;      // 1/|q_t| fp32 [64]
constexpr uint32_t P_RK = P_RQ + 256;      // 1/|k_t|
constexpr uint32_t P_DQK = P_RK + 256;     // q^_t . k^_t
constexpr uint32_t P_TOT = P_DQK + 256;    // half-chunk decay fp32 [2][128]
constexpr uint32_t P_BAR = 98304;          // 10 mbarriers, TMEM slot, the next units
constexpr uint32_t P_LAYOUT = P_BAR + 256;
// 97 KiB per CTA, so that two CTAs (with the 1 KiB each that the system
// keeps) fit the 196 KiB shared-memory carveout and leave the SM 60 KiB of
// L1 (the next carveout, 228 KiB, leaves 28 KiB, less than the two CTAs'
// register-spill slots).  The layout needs 1024-byte alignment: the slack
// covers a dynamic base aligned to 256 bytes; a CTA that finds less reports
// KDA_ERR_ALIGNMENT and leaves.
constexpr uint32_t P_SMEM = 99328;
constexpr int P_CARVEOUT_PCT = 85;         // of 228 KiB, rounded up to the 196 KiB carveout
static_assert(P_TOT + 1024 <= P_TP + 8192, "the small vectors fit in the T' region");
static_assert(P_TF + C * LDA * 4 <= P_XT, "A_kk and T fit below X'^T");
static_assert(P_PAIR + 49152 <= P_XT, "pair-sum operands fit below X'^T");
static_assert(P_LAYOUT + 768 <= P_SMEM, "slack for a 256-byte-aligned base");
static_assert(2 * (P_SMEM + 1024) <= 200704, "two preparation CTAs in the 196 KiB carveout");
constexpr uint32_t P_TM_A = 0, P_TM_W = 0, P_TM_U = 64, P_TM_COLS = 256;

// TMA descriptors of the preparation's inputs, each a [T][H][128] tensor read
// as boxes of 64 rows of one head: q, k, v (16-bit inputs only) and g or f.
struct PrepMaps {
    CUtensorMap q, k, v, g;
};

// Where one (chunk, head) unit lies in the packed input.
struct UnitLoc {
    int64_t unit;
    int32_t valid, h, t0, L;
};

// Persistent: each CTA takes units in order from the window's counter (so CTAs
// that start late, on SMs a scan frees, find the work already shared out) and
// keeps its tensor memory and barriers across them.  The next unit's inputs
// are staged by TMA tile loads while the current one finishes: q, k (and f in
// BF16) as soon as the inverse has freed their region, v (and an FP32 g or f)
// once the W/U MMAs have read X'^T and V^T.
template <typename TIn, int kGate>
__global__ void __launch_bounds__(NT, 2) chunk_prep_kernel(ChunkArgs args,
                                                           const __grid_constant__ PrepMaps maps,
                                                           const int32_t* __restrict__ hdr,
                                                           unsigned char* __restrict__ records,
                                                           int64_t unit_base, int64_t units,
                                                           int32_t* __restrict__ ctr,
                                                           int32_t wait_primary)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    unsigned char* sm = smem_raw + pad;
    const uint32_t sb = raw_s + pad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, half = warp >> 2;
    const int row = 32 * quad + lane;                      // TMEM lane
    const int ch = tid & 127, hh = tid >> 7;               // channel / token-half ownership
    const int H = args.H;

    // A window launched beside the previous window's scan (programmatic
    // dependent launch) completes only after that scan: its last CTA waits for
    // it, so the next scan, launched after this grid, sees the state carry.
    if (wait_primary && blockIdx.x == gridDim.x - 1 && tid == 0) grid_dependency_wait();
    if (pad + P_LAYOUT > P_SMEM) {                         // the same for every CTA
        if (tid == 0) report_status(args.status, KDA_ERR_ALIGNMENT);
        return;
    }
    const int32_t* off = hdr + kHdrOff;

    float (*akk)[LDA] = reinterpret_cast<float (*)[LDA]>(sm + P_AKK);
    float (*Tf)[LDA] = reinterpret_cast<float (*)[LDA]>(sm + P_TF);
    const uint16_t* sq = reinterpret_cast<const uint16_t*>(sm + P_SQ);
    const uint16_t* sk = reinterpret_cast<const uint16_t*>(sm + P_SK);
    const uint16_t* sv = reinterpret_cast<const uint16_t*>(sm + P_SV);
    constexpr bool kGated = kGate != kGateG;
    using TG = typename GateSrc<kGate>::T;                 // element of g or f
    const TG* sg = reinterpret_cast<const TG*>(sm + P_SG);
    float* rq = reinterpret_cast<float*>(sm + P_RQ);
    float* rk = reinterpret_cast<float*>(sm + P_RK);
    float* dqk = reinterpret_cast<float*>(sm + P_DQK);
    float* sbeta = reinterpret_cast<float*>(sm + P_BETA);
    float* tot = reinterpret_cast<float*>(sm + P_TOT);
    // [0..2] pair rounds, [3] W/U, [4] drain after a failure, [5..7] the
    // operands of pair round 0..2 written (every thread arrives)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + P_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + P_BAR + 64);
    // [0] the CTA's first unit, [1] the unit after the current one
    UnitLoc* s_loc = reinterpret_cast<UnitLoc*>(sm + P_BAR + 80);
    // the staging of a unit's inputs: [0] early part, [1] late part (one phase per unit)
    uint64_t* sbar = reinterpret_cast<uint64_t*>(sm + P_BAR + 128);
    // test hook: CTA 0 withholds its first MMA group and the commit that signals it
    const bool withhold = args.fault == KDA_TEST_FAULT_PREP && blockIdx.x == 0;

    const TIn* __restrict__ gq = static_cast<const TIn*>(args.q);
    const TIn* __restrict__ gk = static_cast<const TIn*>(args.k);
    const TIn* __restrict__ gv = static_cast<const TIn*>(args.v);
    const TG* __restrict__ graw =
        kGated ? static_cast<const TG*>(args.f) : reinterpret_cast<const TG*>(args.g);
    using ST = Stage<TIn>;
    constexpr bool k16 = sizeof(TIn) == 2;                 // 16-bit inputs: staged by TMA
    constexpr bool kGEarly = sizeof(TG) == 2;              // a BF16 f fits beside q and k
    constexpr int GP = DK * (int)sizeof(TG) / 16;          // 16-byte pieces per g/f row
    constexpr uint32_t kRow16 = C * DK * 2, kRowG = C * DK * sizeof(TG);   // bytes of one box
    constexpr uint32_t kEarlyBytes = (k16 ? 2 * kRow16 : 0) + (kGEarly ? kRowG : 0);
    constexpr uint32_t kLateBytes = (k16 ? kRow16 : 0) + (kGEarly ? 0 : kRowG);

    // The next unit of this window, taken from its counter and located in the
    // packed input by one thread (its dependent loads of the offsets run while
    // the CTA waits for the current unit's staging); the rest read it after a
    // barrier.
    auto grab_locate = [&](UnitLoc* slot) {
        const int64_t c = atomicAdd(ctr, 1);
        UnitLoc u{unit_base + c, 0, 0, 0, 0};
        const int32_t gc = (int32_t)(u.unit / H);
        if (c < units && gc < off[args.N]) {               // else past the window or the chunks
            int lo = 0, hi = args.N - 1;                   // last n with off[n] <= gc
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (off[mid] <= gc) lo = mid;
                else hi = mid - 1;
            }
            const int bos = args.cu_seqlens[lo], eos = args.cu_seqlens[lo + 1];
            u.valid = 1;
            u.h = (int)(u.unit % H);
            u.t0 = bos + (gc - off[lo]) * C;
            u.L = min(C, eos - u.t0);
        }
        *slot = u;
    };
    // The staging copies, issued by thread 0: 64 rows of one head, dense
    // [64][128] in shared memory.  Rows past the end of the tensor arrive as
    // zeros; rows of the next sequence inside a packed batch are cleared at the
    // top of the unit.  Thread 0 counts the copies of each part issued and
    // waited for (s_cnt: [0, 1] early, [2, 3] late).
    int32_t* s_cnt = reinterpret_cast<int32_t*>(sm + P_BAR + 144);
    // q, k (and a BF16 f): their region is free once the inverse is done
    auto stage_early = [&](const UnitLoc& u) {
        if (tid == 0 && kEarlyBytes > 0) {
            mbar_arrive_expect_tx(&sbar[0], kEarlyBytes);
            if constexpr (k16) {
                tma_load_3d(sm + P_SQ, &maps.q, 0, u.h, u.t0, &sbar[0]);
                tma_load_3d(sm + P_SK, &maps.k, 0, u.h, u.t0, &sbar[0]);
            }
            if constexpr (kGEarly) tma_load_3d(sm + P_SG, &maps.g, 0, u.h, u.t0, &sbar[0]);
            ++s_cnt[0];
        }
    };
    // v (and an FP32 g or f): free once the W/U MMAs have read X'^T and V^T
    auto stage_late = [&](const UnitLoc& u) {
        if (tid == 0 && kLateBytes > 0) {
            mbar_arrive_expect_tx(&sbar[1], kLateBytes);
            if constexpr (k16) tma_load_3d(sm + P_SV, &maps.v, 0, u.h, u.t0, &sbar[1]);
            if constexpr (!kGEarly) tma_load_3d(sm + P_SG, &maps.g, 0, u.h, u.t0, &sbar[1]);
            ++s_cnt[2];
        }
    };

    if (warp == 0) {
        tmem_alloc(tslot, P_TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 8; ++b) mbar_init(&bar[b], b >= 5 ? NT : 1);
        mbar_init(&sbar[0], 1);
        mbar_init(&sbar[1], 1);
        for (int i = 0; i < 4; ++i) s_cnt[i] = 0;
        fence_mbar_init();
        grab_locate(&s_loc[0]);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tlane = tmem + ((uint32_t)(32 * quad) << 16);

    UnitLoc cur = s_loc[0];
    if (cur.valid) {
        stage_early(cur);
        stage_late(cur);
    }
    bool failed = false;
    uint32_t ph = 0;                                       // each barrier completes once per unit
    constexpr uint32_t id_pairs = idesc(kFmtF16, 128, 64, true, true);
    // A pair round: every thread arrives once its operand rows are written, and
    // only the issuing thread waits for the arrivals; the others go on at once.
    auto issue_round = [&](int rnd) {
        fence_async_smem();
        fence_before_sync();
        mbar_arrive(&bar[5 + rnd]);
        if (tid == 0 && !(withhold && rnd == 0)) {
            if (!mbar_wait(&bar[5 + rnd], ph)) {
                failed = true;                             // no commit: the others time out too
            } else {
                fence_after_sync();
                const uint64_t da = desc_mnmajor128(sb + P_PAIR, 16384, 0);
                const uint64_t db = desc_mnmajor64(sb + P_PAIR + 32768, 0);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_f16(tmem + P_TM_A + 64 * rnd, desc_advance(da, mnmajor_off(s)),
                            desc_advance(db, mnmajor_off(s)), id_pairs, s > 0);
                commit(&bar[rnd]);
            }
        }
    };
    // Each thread waits for a round's MMAs before it overwrites their operands;
    // a wait that gives up is only recorded here, and the CTA decides together
    // at the next barrier (a lone thread leaving early would desert the CTA's
    // later barriers).
    auto wait_round = [&](int b) {
        if (!mbar_wait(&bar[b], ph)) failed = true;
    };
    auto wait_bar = [&](int b) -> bool {
        const bool ok = mbar_wait(&bar[b], ph);
        return __syncthreads_or(failed || !ok) == 0;
    };

    while (cur.valid) {
        const int h = cur.h, t0 = cur.t0, L = cur.L;
        unsigned char* rec = records + cur.unit * REC_BYTES;

        // ---- 1: the chunk in staging (rows >= L zero, decay 1)
        if constexpr (!k16) {
            using LD = Loader<TIn>;
            constexpr int P = LD::kPieces;
            auto rows_via_regs = [&](const TIn* base, uint32_t so) {
                uint4 x[C * P / NT];
#pragma unroll
                for (int u = 0; u < C * P / NT; ++u) {
                    const int e = tid + u * NT, r = e / P, pc = e % P;
                    x[u] = (r < L) ? LD::load(base + ((int64_t)(t0 + r) * H + h) * DK, pc)
                                   : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < C * P / NT; ++u) {
                    const int e = tid + u * NT;
                    LD::store(sm + so, e / P, e % P, x[u]);
                }
            };
            rows_via_regs(gq, P_SQ);
            rows_via_regs(gk, P_SK);
            rows_via_regs(gv, P_SV);
        }
        float lamneg = 0.f, dtb = 0.f;
        if (kGated) {
            lamneg = -expf(args.A_log[h]);
            dtb = args.dt_bias[(int64_t)h * DK + ch];
        }
        if (tid < C) {
            float xb = 0.f;
            if (tid < L) {
                const int64_t i = (int64_t)(t0 + tid) * H + h;
                if (kGated)
                    xb = gate_sigmoid(args.b_bf16
                                          ? __bfloat162float(static_cast<const __nv_bfloat16*>(args.b)[i])
                                          : static_cast<const float*>(args.b)[i]);
                else
                    xb = args.beta[i];
            }
            sbeta[tid] = xb;
        }
        if (tid == 4 * 32) grab_locate(&s_loc[1]);          // read after the inverse
        {
            const bool ok_e = kEarlyBytes == 0 || mbar_wait(&sbar[0], ph);
            const bool ok_l = kLateBytes == 0 || mbar_wait(&sbar[1], ph);
            const bool ok = ok_e && ok_l;
            if (tid == 0) {
                if (kEarlyBytes > 0 && ok_e) ++s_cnt[1];
                if (kLateBytes > 0 && ok_l) ++s_cnt[3];
            }
            if (__syncthreads_or(!ok)) { failed = true; break; }
        }
        if (L < C) {
            // the staged rows past the sequence end hold the next sequence's
            // tokens: zero (decay 1)
            if constexpr (k16) {
                for (int e = tid; e < (C - L) * 16; e += NT) {
                    const uint32_t o = (uint32_t)(L + (e >> 4)) * 256 + (e & 15) * 16;
                    *reinterpret_cast<uint4*>(sm + P_SQ + o) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(sm + P_SK + o) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(sm + P_SV + o) = make_uint4(0, 0, 0, 0);
                }
            }
            for (int e = tid; e < (C - L) * GP; e += NT)
                *reinterpret_cast<uint4*>(sm + P_SG + (uint32_t)L * GP * 16 + e * 16) = make_uint4(0, 0, 0, 0);
            __syncthreads();
        }

        // ---- 2: row norms and q^ . k^
        chunk_norms<TIn>(sm + P_SQ, sm + P_SK, rq, rk, dqk, args.l2norm != 0, tid);
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
                    const float gv_ = load_as_float(sg + t * DK + ch);
                    a[u] = kGated ? (t < L ? gate_exp_fast(gv_, dtb, lamneg) : 1.f) : __expf(gv_);
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

        // ---- 4: pair sums, three rounds through one operand buffer; the
        // per-channel rows and the zeroing of A_qk's upper part run beside the MMAs
        float vv[32];
        level32_operands(sm + P_PAIR, ch, hh, a, kh, qh);
        level_operands<16>(sm + P_PAIR, ch, hh, 64, 32, a, kh, qh);
        issue_round(0);
        {
            // X'^T (shared, over the dead g staging), Q' and K''^T (record), d
            const float before = hh ? tot[ch] : 1.f;
            const float after = hh ? 1.f : tot[DK + ch];
            if (hh == 0) reinterpret_cast<float*>(rec + REC_DEC)[ch] = tot[ch] * tot[DK + ch];
            channel_rows(sm + P_XT, rec + REC_QP, rec + REC_KT, ch, hh, before, after, a, kh, qh);
        }
        wait_round(0);
        level_operands<8>(sm + P_PAIR, ch, hh, 0, 0, a, kh, qh);
        level_operands<4>(sm + P_PAIR, ch, hh, 64, 32, a, kh, qh);
        issue_round(1);
        aqk_zero_upper(sm + P_AQK, tid);
        wait_round(1);
        level_operands<2>(sm + P_PAIR, ch, hh, 0, 0, a, kh, qh);
        level_operands<1>(sm + P_PAIR, ch, hh, 64, 32, a, kh, qh);
        issue_round(2);
        // v column of this thread, read before the barrier that precedes the
        // in-place V^T writes (which also settles any wait that gave up)
#pragma unroll
        for (int u = 0; u < 32; ++u) vv[u] = ST::to_f32(sv[(32 * hh + u) * DV + ch]);
        if (!wait_bar(2)) { failed = true; break; }
#pragma unroll
        for (int q = 0; q < 4; ++q) st8(sm + P_SV, 0, ch, 32 * hh + 8 * q, vv + 8 * q);
        fence_after_sync();

        // ---- 5: A_kk (fp32) and A_qk (fp16) from TMEM
        extract_pairs(sm + P_AQK, &akk[0][0], sbeta, dqk, tlane, P_TM_A, tid, warp, lane);
        fence_before_sync();
        __syncthreads();

        // ---- 6: T' = (I + A_kk)^-1 diag(beta)
        chunk_inverse<true>(akk, Tf, sbeta, sm + P_TP, tid, warp, lane);
        fence_async_smem();
        fence_before_sync();
        __syncthreads();
        const UnitLoc nxt = s_loc[1];
        if (nxt.valid) stage_early(nxt);                   // into the dead q, k, f, A_kk, T

        // ---- 7: W^T = X'^T T'^T, U^T = V^T T'^T
        if (tid == 0) {
            fence_after_sync();
            constexpr uint32_t id = idesc(kFmtF16, 128, 64);
            const uint64_t dx = desc_kmajor(sb + P_XT, 128, 0), dv = desc_kmajor(sb + P_SV, 128, 0);
            const uint64_t dt = desc_kmajor(sb + P_TP, 64, 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + P_TM_W, desc_advance(dx, kmajor_off(128, s)),
                        desc_advance(dt, kmajor_off(64, s)), id, s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_f16(tmem + P_TM_U, desc_advance(dv, kmajor_off(128, s)),
                        desc_advance(dt, kmajor_off(64, s)), id, s > 0);
            commit(&bar[3]);
        }
        {
            // A_qk tile to the record while the MMAs run (32 bytes per thread)
            const uint4* src = reinterpret_cast<const uint4*>(sm + P_AQK);
            uint4* dst = reinterpret_cast<uint4*>(rec + REC_AQK);
            dst[tid] = src[tid];
            dst[tid + NT] = src[tid + NT];
        }
        if (!wait_bar(3)) { failed = true; break; }
        fence_after_sync();
        if (nxt.valid) stage_late(nxt);                    // into the read X'^T, V^T
        {
            float w[32];
            tmem_ld32(tlane + P_TM_W + 32 * half, w);
#pragma unroll
            for (int q = 0; q < 4; ++q) st8(rec + REC_W, 0, row, 32 * half + 8 * q, w + 8 * q);
            tmem_ld32(tlane + P_TM_U + 32 * half, w);
#pragma unroll
            for (int q = 0; q < 4; ++q) st8(rec + REC_U, 0, row, 32 * half + 8 * q, w + 8 * q);
        }
        cur = nxt;
        ph ^= 1u;
    }

    if (failed && tid == 0) {
        report_status(args.status, KDA_ERR_TIMEOUT);
        // every MMA this thread issued finishes before the TMEM is released
        commit(&bar[4]);
        mbar_wait(&bar[4], 0);
    }
    // the staging of a next unit, if any, lands before the CTA leaves
    if (tid == 0 && s_cnt[0] > s_cnt[1]) mbar_wait(&sbar[0], (s_cnt[0] - 1) & 1);
    if (tid == 0 && s_cnt[2] > s_cnt[3]) mbar_wait(&sbar[1], (s_cnt[2] - 1) & 1);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, P_TM_COLS);
}

// ---------------------------------------------------------------- scan
// One CTA per (sequence, head): eight epilogue warps (thread = state row v and
// a half of the columns) and one control warp whose lane 0 issues the bulk
// copies and the MMAs.  Per chunk c (TMEM region R = 256 (c & 1)):
//   control:  record c in stage c & 1 (bulk copy, issued a chunk ahead)
//             [W S]^T -> R (8 MMAs, N = 64), commit ws_done; [Q' S]^T -> R + 64
//   epilogue: Delta^T = U^T - [W S]^T -> shared (fp16), arrive delta_ready
//   control:  P^T = Delta^T K'' (4 MMAs, N = 128), commit p_done; then
//             O^T += Delta^T A_qk^T on top of Q' S (4 MMAs, N = 64), commit o_done
//   epilogue: S^T <- S^T Diag(d) + P^T and the fp16 copy of S^T for the next
//             chunk; arrive s_ready; then O read from TMEM once o_done has
//             come, arrive o_read, and chunk c's output rows, stored while the
//             control warp issues chunk c + 1's MMAs into the other region
// so the state's chain per chunk is [W S] -> Delta -> P -> S: two short MMA
// groups and two short epilogues; Q' S and A_qk Delta ride behind them.  The
// control waits for o_read of chunk c - 2 before it writes region (c & 1)
// again (one barrier per chunk parity), and for o_done of chunk c - 1 before
// it refills that chunk's record stage.
constexpr int SCAN_THREADS = NT + 32;
constexpr int kL2Ahead = 4;                   // records prefetched into L2 this many chunks ahead
constexpr uint32_t kEpiBar = 1;               // named barrier of the 256 epilogue threads
constexpr uint32_t S_ST = 0;                  // S^T fp16 K-major [128 v][128 c]
constexpr uint32_t S_DT = 32768;              // Delta^T fp16 K-major [128 v][64 i]
constexpr uint32_t S_STG = 49152;             // two record stages
constexpr uint32_t S_STG_STRIDE = 74752;      // REC_BYTES rounded up to 1024
constexpr uint32_t S_BAR = S_STG + 2 * S_STG_STRIDE;   // 8 mbarriers, TMEM slot, abort flag
constexpr uint32_t S_SMEM = S_BAR + 128 + 1024;
// With the output gate fused (kNorm): the chunk's z rows (BF16 [64 t][128 v])
// and the per-warp partial sums of squares ([2 halves][4 quads][32 tokens]).
constexpr uint32_t S_Z = S_BAR + 1024;
constexpr uint32_t S_RED = S_Z + 16384;
constexpr uint32_t S_SMEM_NORM = S_RED + 1024 + 1024;
static_assert(S_SMEM_NORM <= 232448, "shared memory budget with the output gate");
static_assert(S_STG_STRIDE >= REC_BYTES && S_STG_STRIDE % 1024 == 0, "stage alignment");
static_assert(S_SMEM <= 232448, "shared memory budget");
// TMEM region of one parity: [W S]^T, O^T (on top of [Q' S]^T), P^T.
constexpr uint32_t S_TM_WS = 0, S_TM_O = 64, S_TM_P = 128, S_TM_REGION = 256, S_TM_COLS = 512;

__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// The scan of the chunks whose global index lies in [g0, g1): a sequence
// whose chunks span several windows enters each later window with the state
// the previous one left in `carry` ([N,H,K,V] FP32, workspace).  The window
// holding a sequence's last chunk (for an empty sequence, the last window)
// writes its final state.
struct ScanWindow {
    int32_t g0, g1;
    float* carry;
    int32_t last;
};

// Sum over the 32 lanes of a warp of each of 32 values, scattered: lane l
// returns the sum of every lane's v[l] (five halving steps, 31 shuffles).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < off; ++k) {
            const float send = upper ? v[k] : v[k + off];
            const float keep = upper ? v[k + off] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0];
}

template <typename TOut, bool kNorm>
__global__ void __launch_bounds__(SCAN_THREADS, 1) chunk_scan_kernel(ChunkArgs args,
                                                                     const int32_t* __restrict__ hdr,
                                                                     const unsigned char* __restrict__ records,
                                                                     ScanWindow win)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
    unsigned char* sm = smem_raw + pad;
    const uint32_t sb = raw_s + pad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool ctrl = warp == NT / 32;
    const int quad = warp & 3, half = (warp >> 2) & 1;
    const int row = 32 * quad + lane;                      // TMEM lane = state row v
    const int H = args.H;
    const int n = hdr[kHdrOff + args.N + 1 + blockIdx.x / H], h = blockIdx.x % H;
    // the next preparation window may start on the SMs this grid leaves free
    launch_dependents();

    const int eos = args.cu_seqlens[n + 1];
    int bos = args.cu_seqlens[n];
    if (bos < 0 || eos < bos || (int64_t)eos > args.T) return;   // reported by the plan
    const int nch_all = (eos - bos + C - 1) / C;
    const int offn = hdr[kHdrOff + n];
    if (offn + nch_all > split_chunk_bound(args.N, args.T)) return;   // bad offsets elsewhere
    const int cb = min(max(win.g0 - offn, 0), nch_all), ce = min(max(win.g1 - offn, 0), nch_all);
    const bool writes_final = (cb < ce && ce == nch_all) || (nch_all == 0 && win.last);
    if (cb == ce && !writes_final) return;                 // no chunk of this sequence here
    const float* state_in = cb == 0 ? args.initial_state : win.carry;
    float* state_out = writes_final ? args.final_state : win.carry;
    bos += cb * C;                                         // the window's chunks, from 0
    const int nch = ce - cb;
    const int64_t rstride = (int64_t)H * REC_BYTES;
    const unsigned char* rec0 = records + ((int64_t)(offn + cb) * H + h) * REC_BYTES;
    TOut* __restrict__ out = static_cast<TOut*>(args.out);
    // [0,1] record stages, [2] ws_done, [3] p_done, [4] delta_ready (NT),
    // [5] s_ready (NT), [6] drain after a failure, [7] o_done, [8,9] o_read of
    // even and odd chunks (NT)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + S_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + S_BAR + 80);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(sm + S_BAR + 84);

    // ---- the entering state (zero, or the caller's)
    float S[64];                                           // S^T[row][64 half + c]
    if (!ctrl) {
        if (state_in != nullptr) {
            const float* s0 = state_in + ((int64_t)n * H + h) * DK * DV;
#pragma unroll
            for (int u = 0; u < 64; ++u) S[u] = s0[(int64_t)(64 * half + u) * DV + row];
        } else {
#pragma unroll
            for (int u = 0; u < 64; ++u) S[u] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(sm + S_ST + sw128_tile(128, row, (64 * half + 8 * q) * 2)) =
                pack_h8(S + 8 * q);
    }
    if (warp == 0) {
        tmem_alloc(tslot, S_TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 10; ++b) mbar_init(&bar[b], (b == 4 || b == 5 || b >= 8) ? NT : 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tlane = tmem + ((uint32_t)(32 * quad) << 16);

    // A bounded wait that also gives up once the other role has.
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
            auto issue_load = [&](int c) {
                unsigned char* stage = sm + S_STG + (c & 1) * S_STG_STRIDE;
                mbar_arrive_expect_tx(&bar[c & 1], REC_BYTES);
                bulk_g2s(stage, rec0 + c * rstride, REC_BYTES, &bar[c & 1]);
            };
            for (int c = 0; c < min(2, nch); ++c) issue_load(c);
            for (int c = 2; c < min(kL2Ahead, nch); ++c) bulk_prefetch_l2(rec0 + c * rstride, REC_BYTES);
            int issued = min(2, nch), c = 0;
            bool fail = false, any_mma = false;
            constexpr uint32_t id_ws = idesc(kFmtF16, 128, 64, false, true);
            constexpr uint32_t id_p = idesc(kFmtF16, 128, 128);
            constexpr uint32_t id_o = idesc(kFmtF16, 128, 64);
            // operand descriptors at k-step 0, computed once (stage 0 and 1)
            const uint64_t dS = desc_kmajor(sb + S_ST, 128, 0), dDt = desc_kmajor(sb + S_DT, 128, 0);
            const uint32_t st0 = sb + S_STG, st1 = sb + S_STG + S_STG_STRIDE;
            const uint64_t dW0 = desc_mnmajor64(st0 + REC_W, 0), dW1 = desc_mnmajor64(st1 + REC_W, 0);
            const uint64_t dQ0 = desc_mnmajor64(st0 + REC_QP, 0), dQ1 = desc_mnmajor64(st1 + REC_QP, 0);
            const uint64_t dK0 = desc_kmajor(st0 + REC_KT, 128, 0), dK1 = desc_kmajor(st1 + REC_KT, 128, 0);
            const uint64_t dA0 = desc_kmajor(st0 + REC_AQK, 64, 0), dA1 = desc_kmajor(st1 + REC_AQK, 64, 0);
            for (; c < nch; ++c) {
                const uint32_t R = tmem + S_TM_REGION * (c & 1);
                // chunk c - 1's state is current; chunk c - 2's O has left region (c & 1)
                if (c > 0 && !wait_or_abort(&bar[5], (c - 1) & 1)) { fail = true; break; }
                if (c > 0 && c + 1 < nch) {
                    // stage (c + 1) & 1 held chunk c - 1, whose last MMA group
                    // (A_qk Delta, signalled by o_done, done by now in practice)
                    // must be done reading it; the copy then has this chunk's
                    // whole chain to land
                    if (!wait_or_abort(&bar[7], (c - 1) & 1)) { fail = true; break; }
                    issue_load(c + 1);
                    issued = c + 2;
                }
                if (c > 1 && !wait_or_abort(&bar[8 + (c & 1)], ((c - 2) >> 1) & 1)) { fail = true; break; }
                if (!wait_or_abort(&bar[c & 1], (c >> 1) & 1)) { fail = true; break; }
                fence_after_sync();
                const bool odd = c & 1;
                const uint64_t dW = odd ? dW1 : dW0, dQ = odd ? dQ1 : dQ0;
                const uint64_t dK = odd ? dK1 : dK0, dA = odd ? dA1 : dA0;
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_f16(R + S_TM_WS, desc_advance(dS, kmajor_off(128, s)),
                            desc_advance(dW, mnmajor_off(s)), id_ws, s > 0);
                commit(&bar[2]);
                any_mma = true;
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_f16(R + S_TM_O, desc_advance(dS, kmajor_off(128, s)),
                            desc_advance(dQ, mnmajor_off(s)), id_ws, s > 0);
                if (c + kL2Ahead < nch) bulk_prefetch_l2(rec0 + (c + kL2Ahead) * rstride, REC_BYTES);
                if (!wait_or_abort(&bar[4], c & 1)) { fail = true; break; }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(R + S_TM_P, desc_advance(dDt, kmajor_off(128, s)),
                            desc_advance(dK, kmajor_off(128, s)), id_p, s > 0);
                commit(&bar[3]);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(R + S_TM_O, desc_advance(dDt, kmajor_off(128, s)),
                            desc_advance(dA, kmajor_off(64, s)), id_o, 1);
                commit(&bar[7]);
            }
            if (fail) {
                *abort_flag = 1;
                report_status(args.status, KDA_ERR_TIMEOUT);
                // let the MMAs and copies in flight finish before the CTA leaves
                if (any_mma) {
                    commit(&bar[6]);
                    mbar_wait(&bar[6], 0);
                }
                for (int cc = c; cc < issued; ++cc) mbar_wait(&bar[cc & 1], (cc >> 1) & 1);
            }
        }
    } else {
        // out rows of chunk cc = scale O (o: this thread's 32 tokens of its V
        // column, read from TMEM), stored straight from registers: each store
        // instruction writes 32 consecutive V values of one token.  `nan_acc`
        // gathers x * 0 over every stored value: it turns NaN once one of them
        // is infinite or NaN (an FP16 operand out of range, or a bad input).
        float nan_acc = 0.f;
        auto store_chunk_out = [&](int cc, const float (&o)[32]) {
            const int tc = bos + cc * C, Lc = min(C, eos - tc);
            const int64_t ostride = (int64_t)H * DV;
            TOut* op = out + ((int64_t)(tc + 32 * half) * H + h) * DV + row;
            const int nrows = min(32, Lc - 32 * half);
            float y[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) y[u] = args.scale * o[u];
            if constexpr (kNorm) {
                // y = o / sqrt(mean_v o^2 + eps) * w[v] * sigmoid(z): the sum of
                // squares of token 32 half + u over v is spread over the 128
                // threads of this half (lanes of four warps); each warp sums its
                // 32 v values per token (lane u ends with token u), the four
                // warps' sums meet in shared memory, and each lane's 1/rms goes
                // back to the lanes by shuffles.
                float sq[32];
#pragma unroll
                for (int u = 0; u < 32; ++u) sq[u] = y[u] * y[u];
                float* red = reinterpret_cast<float*>(sm + S_RED);
                red[(half * 4 + quad) * 32 + lane] = warp_reduce_scatter32(sq, lane);
                cp_async_wait_all();                   // this chunk's z rows
                named_sync(kEpiBar, NT);
                const float ss = red[(half * 4) * 32 + lane] + red[(half * 4 + 1) * 32 + lane] +
                                 red[(half * 4 + 2) * 32 + lane] + red[(half * 4 + 3) * 32 + lane];
                const float rstd = rsqrtf(ss * (1.f / DV) + args.norm_eps);
                const float wv = args.norm_w[row];
                const __nv_bfloat16* zt = reinterpret_cast<const __nv_bfloat16*>(sm + S_Z);
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const float zv = __bfloat162float(zt[(32 * half + u) * DV + row]);
                    const float gate = __fdividef(1.f, 1.f + __expf(-zv));
                    y[u] *= __shfl_sync(0xffffffffu, rstd, u) * wv * gate;
                }
            }
#pragma unroll
            for (int u = 0; u < 32; ++u) {
                if (u < nrows) {
                    nan_acc = fmaf(y[u], 0.f, nan_acc);
                    store_out(op, y[u]);
                }
                op += ostride;
            }
        };
        // the z rows of chunk cc into the tile (rows past the sequence end zero)
        auto stage_z = [&](int cc) {
            const int tc = bos + cc * C, Lc = min(C, eos - tc);
#pragma unroll
            for (int k = 0; k < C * 16 / NT; ++k) {
                const int e = tid + k * NT, r = e >> 4, pc = e & 15;
                const bool ok = r < Lc;
                cp_async16(sm + S_Z + r * 256 + pc * 16,
                           args.z + ((int64_t)(tc + (ok ? r : 0)) * H + h) * DV + pc * 8, ok);
            }
            cp_async_commit();
        };
        // test hook: CTA 0 withholds its first delta_ready arrival
        const bool withhold = args.fault == KDA_TEST_FAULT_SCAN && blockIdx.x == 0;
        bool fail = false;
        for (int c = 0; c < nch; ++c) {
            const uint32_t R = tlane + S_TM_REGION * (c & 1);
            unsigned char* stage = sm + S_STG + (c & 1) * S_STG_STRIDE;
            uint4 u4[4];                                   // this thread's U^T row piece
            {
                bool ok = wait_or_abort(&bar[c & 1], (c >> 1) & 1);
                if (ok) {
                    const unsigned char* up = stage + REC_U;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        u4[q] = *reinterpret_cast<const uint4*>(up + sw128(row, (32 * half + 8 * q) * 2));
                    ok = wait_or_abort(&bar[2], c & 1);
                }
                if (named_sync_or(kEpiBar, NT, !ok)) { fail = true; break; }
            }
            // every epilogue thread is past chunk c - 1's outputs: its z tile is free
            if constexpr (kNorm) stage_z(c);
            fence_after_sync();
            {
                // Delta^T[v][i] = U^T[v][i] - [W S]^T[v][i], fp16 K-major
                float ws[32], d[8];
                tmem_ld32(R + S_TM_WS + 32 * half, ws);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t w4[4] = {u4[q].x, u4[q].y, u4[q].z, u4[q].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 uf = __half22float2(*reinterpret_cast<const __half2*>(&w4[e]));
                        d[2 * e] = uf.x - ws[8 * q + 2 * e];
                        d[2 * e + 1] = uf.y - ws[8 * q + 2 * e + 1];
                    }
                    st8(sm + S_DT, 0, row, 32 * half + 8 * q, d);
                }
            }
            fence_async_smem();
            fence_before_sync();
            if (!(withhold && c == 0)) mbar_arrive(&bar[4]);
            {
                const bool ok = wait_or_abort(&bar[3], c & 1);
                if (named_sync_or(kEpiBar, NT, !ok)) { fail = true; break; }
            }
            fence_after_sync();
            {
                // S^T <- S^T Diag(d) + P^T;  fp16 copy of S^T
                const float4* dec4 = reinterpret_cast<const float4*>(stage + REC_DEC) + 16 * half;
                float p[32];
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    tmem_ld32(R + S_TM_P + 64 * half + 32 * part, p);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float4 f = dec4[8 * part + u];
                        float* sv = S + 32 * part + 4 * u;
                        sv[0] = sv[0] * f.x + p[4 * u + 0];
                        sv[1] = sv[1] * f.y + p[4 * u + 1];
                        sv[2] = sv[2] * f.z + p[4 * u + 2];
                        sv[3] = sv[3] * f.w + p[4 * u + 3];
                    }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<uint4*>(sm + S_ST + sw128_tile(128, row, (64 * half + 8 * q) * 2)) =
                        pack_h8(S + 8 * q);
            }
            // the next chunk's MMAs may start (into the other region) while this
            // chunk's O is read
            fence_async_smem();
            fence_before_sync();
            mbar_arrive(&bar[5]);
            {
                const bool ok = wait_or_abort(&bar[7], c & 1);
                if (named_sync_or(kEpiBar, NT, !ok)) { fail = true; break; }
            }
            fence_after_sync();
            float o[32];
            tmem_ld32(R + S_TM_O + 32 * half, o);
            fence_before_sync();
            mbar_arrive(&bar[8 + (c & 1)]);
            // its rows go out while the control warp issues the next chunk's MMAs
            store_chunk_out(c, o);
        }
        if (fail) {
            *abort_flag = 1;
            if (tid == 0) report_status(args.status, KDA_ERR_TIMEOUT);
        } else if (state_out != nullptr) {
            float* fs = state_out + ((int64_t)n * H + h) * DK * DV;
#pragma unroll
            for (int u = 0; u < 64; ++u) {
                nan_acc = fmaf(S[u], 0.f, nan_acc);
                fs[(int64_t)(64 * half + u) * DV + row] = S[u];
            }
        }
        if (nan_acc != nan_acc) report_status(args.status, KDA_ERR_RANGE);
    }
    if constexpr (kNorm) cp_async_wait_all();
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, S_TM_COLS);
}

// 32 consecutive output values of one row (16-byte stores; the row piece is
// 64-byte aligned for BF16 and 128-byte aligned for FP32).
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
        uint4 w;
        uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[8 * q + 2 * e], o[8 * q + 2 * e + 1]);
            wp[e] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        reinterpret_cast<uint4*>(p)[q] = w;
    }
}

// ---------------------------------------------------------------- scan, V in halves
// The recurrence is separable in the columns of the state (every column of S
// evolves with the same W, Q', K'', A_qk and decay, and only its own column of
// U), so each (sequence, head) is scanned by two CTAs, one per half of V (64
// columns each).  Per chunk c, in TMEM region R = 128 (c & 1):
//   control:  D1 = [W; Q'] S_v (8 MMAs, M = 128: rows 0..63 W S, 64..127 Q' S),
//             commit d1_done
//   epilogue (warps of lanes 0..63): Delta = U_v - W S_v -> shared (fp16),
//             arrive delta_ready
//   control:  P = K''^T Delta (4 MMAs) into R + 64, commit p_done; then
//             D1 += [any; A_qk] Delta (4 MMAs; its rows 0..63 are dead), commit
//             o_done
//   epilogue (all warps): S_v <- Diag(d) S_v + P and its fp16 copy, arrive
//             s_ready; then the warps of lanes 64..127 read O once o_done has
//             come, arrive o_read and store the chunk's outputs
// so the state's chain per chunk is D1 -> Delta -> P -> S, with half the
// columns of the full-width scan per CTA.  The control warp waits for o_read
// of chunk c - 2 before it writes region (c & 1) again, and for o_done of
// chunk c - 1 before it refills that chunk's record stage.  o_read has one
// barrier per chunk parity: the O warps may have finished chunk c - 1 as well
// when the control asks about chunk c - 2, and a single barrier two phases
// ahead of its waiter would make the parity wait ambiguous.
constexpr int VH = 64;                        // state columns per CTA
constexpr uint32_t V_ST = 0;                  // S_v fp16 MN-major [128 c][64 v]
constexpr uint32_t V_DT = 16384;              // Delta fp16 MN-major [64 i][64 v]
constexpr uint32_t V_STG = 24576;             // two record stages
constexpr uint32_t V_BAR = V_STG + 2 * S_STG_STRIDE;   // 10 mbarriers, TMEM slot, abort flag
constexpr uint32_t V_SMEM = V_BAR + 128 + 1024;
static_assert(V_SMEM <= 232448, "shared memory budget of the V-half scan");
constexpr uint32_t V_TM_D1 = 0, V_TM_P = 64, V_TM_REGION = 128, V_TM_COLS = 256;
constexpr uint32_t kDeltaBar = 2;             // named barrier of the four Delta warps

template <typename TOut>
__global__ void __launch_bounds__(SCAN_THREADS, 1) chunk_scan_vh_kernel(ChunkArgs args,
                                                                        const int32_t* __restrict__ hdr,
                                                                        const unsigned char* __restrict__ records,
                                                                        ScanWindow win)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
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
    const int vh = blockIdx.x & 1;                         // this CTA's half of V
    const int hb = blockIdx.x >> 1;
    const int n = hdr[kHdrOff + args.N + 1 + hb / H], h = hb % H;
    launch_dependents();

    const int eos = args.cu_seqlens[n + 1];
    int bos = args.cu_seqlens[n];
    if (bos < 0 || eos < bos || (int64_t)eos > args.T) return;   // reported by the plan
    const int nch_all = (eos - bos + C - 1) / C;
    const int offn = hdr[kHdrOff + n];
    if (offn + nch_all > split_chunk_bound(args.N, args.T)) return;   // bad offsets elsewhere
    const int cb = min(max(win.g0 - offn, 0), nch_all), ce = min(max(win.g1 - offn, 0), nch_all);
    const bool writes_final = (cb < ce && ce == nch_all) || (nch_all == 0 && win.last);
    if (cb == ce && !writes_final) return;
    const float* state_in = cb == 0 ? args.initial_state : win.carry;
    float* state_out = writes_final ? args.final_state : win.carry;
    bos += cb * C;
    const int nch = ce - cb;
    const int64_t rstride = (int64_t)H * REC_BYTES;
    const unsigned char* rec0 = records + ((int64_t)(offn + cb) * H + h) * REC_BYTES;
    TOut* __restrict__ out = static_cast<TOut*>(args.out);
    const int v0 = VH * vh + 32 * half;                    // this thread's first column of V
    // [0,1] record stages, [2] d1_done, [3] p_done, [4] delta_ready (128),
    // [5] s_ready (NT), [6] drain after a failure, [7] o_done, [8,9] o_read of
    // even and odd chunks (128)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + V_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + V_BAR + 80);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(sm + V_BAR + 84);

    // ---- the entering state: S[c][v0 .. v0 + 31] of state row c = this thread's lane
    float S[32];
    if (!ctrl) {
        if (state_in != nullptr) {
            const float4* s0 = reinterpret_cast<const float4*>(
                state_in + (((int64_t)n * H + h) * DK + row) * DV + v0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = s0[q];
                S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int u = 0; u < 32; ++u) S[u] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) st8(sm + V_ST, 0, row, 32 * half + 8 * q, S + 8 * q);
    }
    if (warp == 0) {
        tmem_alloc(tslot, V_TM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 10; ++b)
            mbar_init(&bar[b], (b == 4 || b >= 8) ? NT / 2 : b == 5 ? NT : 1);
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
            auto issue_load = [&](int c) {
                unsigned char* stage = sm + V_STG + (c & 1) * S_STG_STRIDE;
                mbar_arrive_expect_tx(&bar[c & 1], REC_BYTES);
                bulk_g2s(stage, rec0 + c * rstride, REC_BYTES, &bar[c & 1]);
            };
            for (int c = 0; c < min(2, nch); ++c) issue_load(c);
            for (int c = 2; c < min(kL2Ahead, nch); ++c) bulk_prefetch_l2(rec0 + c * rstride, REC_BYTES);
            int issued = min(2, nch), c = 0;
            bool fail = false, any_mma = false;
            constexpr uint32_t id_d1 = idesc(kFmtF16, 128, VH, true, true);
            constexpr uint32_t id_pv = idesc(kFmtF16, 128, VH, false, true);
            // operand descriptors at k-step 0, computed once (stage 0 and 1)
            const uint64_t dS = desc_mnmajor64(sb + V_ST, 0), dDl = desc_mnmajor64(sb + V_DT, 0);
            const uint32_t st0 = sb + V_STG, st1 = sb + V_STG + S_STG_STRIDE;
            const uint64_t dW0 = desc_mnmajor128(st0 + REC_W, 16384, 0);
            const uint64_t dW1 = desc_mnmajor128(st1 + REC_W, 16384, 0);
            const uint64_t dK0 = desc_kmajor(st0 + REC_KT, 128, 0), dK1 = desc_kmajor(st1 + REC_KT, 128, 0);
            const uint64_t dA0 = desc_kmajor(st0 + REC_AQK - 8192, 128, 0);
            const uint64_t dA1 = desc_kmajor(st1 + REC_AQK - 8192, 128, 0);
            for (; c < nch; ++c) {
                const uint32_t R = tmem + V_TM_REGION * (c & 1);
                // chunk c - 1's state is current; chunk c - 2's O has left region (c & 1)
                if (c > 0 && !wait_or_abort(&bar[5], (c - 1) & 1)) { fail = true; break; }
                if (c > 0 && c + 1 < nch) {
                    // stage (c + 1) & 1 held chunk c - 1, whose last MMA group
                    // (A_qk Delta, signalled by o_done) must be done reading it;
                    // the copy then has this chunk's whole chain to land
                    if (!wait_or_abort(&bar[7], (c - 1) & 1)) { fail = true; break; }
                    issue_load(c + 1);
                    issued = c + 2;
                }
                if (c > 1 && !wait_or_abort(&bar[8 + (c & 1)], ((c - 2) >> 1) & 1)) { fail = true; break; }
                if (!wait_or_abort(&bar[c & 1], (c >> 1) & 1)) { fail = true; break; }
                fence_after_sync();
                const bool odd = c & 1;
                const uint64_t dW = odd ? dW1 : dW0, dK = odd ? dK1 : dK0, dA = odd ? dA1 : dA0;
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_f16(R + V_TM_D1, desc_advance(dW, mnmajor_off(s)),
                            desc_advance(dS, mnmajor_off(s)), id_d1, s > 0);
                commit(&bar[2]);
                any_mma = true;
                if (c + kL2Ahead < nch) bulk_prefetch_l2(rec0 + (c + kL2Ahead) * rstride, REC_BYTES);
                if (!wait_or_abort(&bar[4], c & 1)) { fail = true; break; }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(R + V_TM_P, desc_advance(dK, kmajor_off(128, s)),
                            desc_advance(dDl, mnmajor_off(s)), id_pv, s > 0);
                commit(&bar[3]);
                // rows 0..63 of this A operand are the 8 KiB before A_qk in the
                // record (finite FP16 values of U^T); they add into the dead W S rows
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_f16(R + V_TM_D1, desc_advance(dA, kmajor_off(128, s)),
                            desc_advance(dDl, mnmajor_off(s)), id_pv, 1);
                commit(&bar[7]);
            }
            if (fail) {
                *abort_flag = 1;
                report_status(args.status, KDA_ERR_TIMEOUT);
                if (any_mma) {
                    commit(&bar[6]);
                    mbar_wait(&bar[6], 0);
                }
                for (int cc = c; cc < issued; ++cc) mbar_wait(&bar[cc & 1], (cc >> 1) & 1);
            }
        }
    } else {
        float nan_acc = 0.f;
        // test hook: CTA 0 withholds its first delta_ready arrival
        const bool withhold = args.fault == KDA_TEST_FAULT_SCAN && blockIdx.x == 0;
        bool fail = false;
        for (int c = 0; c < nch; ++c) {
            const uint32_t R = tlane + V_TM_REGION * (c & 1);
            unsigned char* stage = sm + V_STG + (c & 1) * S_STG_STRIDE;
            __half2 u2[16];                                // U[i][v0 .. v0 + 31] (Delta warps)
            {
                // (an O warp that gave up on the previous chunk carries `fail` here)
                const bool ok = !fail && wait_or_abort(&bar[c & 1], (c >> 1) & 1);
                if (named_sync_or(kEpiBar, NT, !ok)) { fail = true; break; }
            }
            if (dwarp) {
                // U from the record's U^T [v][i] tile, read down a column while D1 runs
                const unsigned char* up = stage + REC_U;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const __half lo = *reinterpret_cast<const __half*>(up + sw128(v0 + 2 * u, 2 * row));
                    const __half hi = *reinterpret_cast<const __half*>(up + sw128(v0 + 2 * u + 1, 2 * row));
                    u2[u] = __halves2half2(lo, hi);
                }
                bool ok = wait_or_abort(&bar[2], c & 1);
                if (named_sync_or(kDeltaBar, NT / 2, !ok)) {
                    fail = true;                           // the others see the abort flag
                } else {
                    fence_after_sync();
                    // Delta[i][v] = U[i][v] - (W S)[i][v], fp16 MN-major
                    float ws[32], dl[32];
                    tmem_ld32(R + V_TM_D1 + 32 * half, ws);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float2 uf = __half22float2(u2[u]);
                        dl[2 * u] = uf.x - ws[2 * u];
                        dl[2 * u + 1] = uf.y - ws[2 * u + 1];
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) st8(sm + V_DT, 0, row, 32 * half + 8 * q, dl + 8 * q);
                    fence_async_smem();
                    fence_before_sync();
                    if (!(withhold && c == 0)) mbar_arrive(&bar[4]);
                }
            }
            {
                const bool ok = !fail && wait_or_abort(&bar[3], c & 1);
                if (named_sync_or(kEpiBar, NT, !ok)) { fail = true; break; }
            }
            fence_after_sync();
            {
                // S_v <- Diag(d) S_v + P;  fp16 copy of S_v for the next chunk
                const float dc = reinterpret_cast<const float*>(stage + REC_DEC)[row];
                float p[32];
                tmem_ld32(R + V_TM_P + 32 * half, p);
#pragma unroll
                for (int u = 0; u < 32; ++u) S[u] = fmaf(S[u], dc, p[u]);
#pragma unroll
                for (int q = 0; q < 4; ++q) st8(sm + V_ST, 0, row, 32 * half + 8 * q, S + 8 * q);
            }
            fence_async_smem();
            fence_before_sync();
            mbar_arrive(&bar[5]);
            if (!dwarp) {
                // O rows (token i = row - 64) leave TMEM, then go out from registers
                const bool ok = wait_or_abort(&bar[7], c & 1);
                float o[32];
                if (ok) {
                    fence_after_sync();
                    tmem_ld32(R + V_TM_D1 + 32 * half, o);
                    fence_before_sync();
                    mbar_arrive(&bar[8 + (c & 1)]);
                    const int i = row - 64, t = bos + c * C + i;
                    if (t < eos) {
                        TOut* op = out + ((int64_t)t * H + h) * DV + v0;
#pragma unroll
                        for (int u = 0; u < 32; ++u) {
                            o[u] *= args.scale;
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
        } else if (state_out != nullptr) {
            float4* fs = reinterpret_cast<float4*>(state_out + (((int64_t)n * H + h) * DK + row) * DV + v0);
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
    if (warp == 0) tmem_dealloc(tmem, V_TM_COLS);
}

// ---------------------------------------------------------------- launch
// cuTensorMapEncodeTiled from the driver (through the runtime, so the library
// needs no link to it); null when the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled()
{
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The descriptor of a [T][H][128] tensor (BF16 or FP32, dense rows) read as
// boxes of 64 tokens x 1 head x 128 values; reads past T return zeros.
cudaError_t encode_rows(CUtensorMap* m, const void* base, bool bf16, int64_t T, int32_t H)
{
    const EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return cudaErrorNotSupported;
    const uint32_t es = bf16 ? 2 : 4;
    const cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)DK * es, (cuuint64_t)H * DK * es};
    const cuuint32_t box[3] = {(cuuint32_t)DK, 1, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                          const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The preparation's descriptors for this call: q, k, v when they are 16-bit
// (FP32 inputs are read through registers), and g or f.
cudaError_t make_prep_maps(const ChunkArgs& a, PrepMaps* maps)
{
    memset(maps, 0, sizeof(*maps));
    cudaError_t e = cudaSuccess;
    if (a.qkv_bf16) {
        e = encode_rows(&maps->q, a.q, true, a.T, a.H);
        if (e == cudaSuccess) e = encode_rows(&maps->k, a.k, true, a.T, a.H);
        if (e == cudaSuccess) e = encode_rows(&maps->v, a.v, true, a.T, a.H);
    }
    if (e != cudaSuccess) return e;
    switch (gate_in(a)) {
        case kGateF32: return encode_rows(&maps->g, a.f, false, a.T, a.H);
        case kGateBF16: return encode_rows(&maps->g, a.f, true, a.T, a.H);
        default: return encode_rows(&maps->g, a.g, false, a.T, a.H);
    }
}

template <typename TIn, int kGate>
cudaError_t launch_prep_typed(const ChunkArgs& a, const PrepMaps& maps, const int32_t* hdr,
                              unsigned char* rec, int64_t unit_base, int64_t units, int32_t* ctr,
                              bool beside_scan, cudaStream_t stream)
{
    auto kern = chunk_prep_kernel<TIn, kGate>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)P_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 P_CARVEOUT_PCT);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count();
    const int64_t ctas = std::min<int64_t>(units, 2 * (int64_t)(sms > 0 ? sms : 152));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = P_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = beside_scan ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a, maps, hdr, rec, unit_base, units, ctr,
                              (int32_t)(beside_scan ? 1 : 0));
}

// Preparation of the (chunk, head) units [unit_base, unit_base + units), taken
// from the counter `ctr` (zero at launch); `beside_scan`: launched to overlap
// the scan just before it on the stream.
cudaError_t launch_prep(const ChunkArgs& a, const PrepMaps& maps, const int32_t* hdr,
                        unsigned char* rec, int64_t unit_base, int64_t units, int32_t* ctr,
                        bool beside_scan, cudaStream_t stream)
{
    if (units <= 0) return cudaSuccess;
#define KDA_PREP(TIN, GATE) \
    launch_prep_typed<TIN, GATE>(a, maps, hdr, rec, unit_base, units, ctr, beside_scan, stream)
    switch (gate_in(a)) {
        case kGateF32:
            return a.qkv_bf16 ? KDA_PREP(__nv_bfloat16, kGateF32) : KDA_PREP(float, kGateF32);
        case kGateBF16:
            return a.qkv_bf16 ? KDA_PREP(__nv_bfloat16, kGateBF16) : KDA_PREP(float, kGateBF16);
        default:
            return a.qkv_bf16 ? KDA_PREP(__nv_bfloat16, kGateG) : KDA_PREP(float, kGateG);
    }
#undef KDA_PREP
}

cudaError_t launch_scan(const ChunkArgs& a, const int32_t* hdr, const unsigned char* rec,
                        ScanWindow win, bool halves, cudaStream_t stream)
{
    if (halves) {
        // plain output: two CTAs per (sequence, head), one per half of V
        auto kv = a.out_bf16 ? chunk_scan_vh_kernel<__nv_bfloat16> : chunk_scan_vh_kernel<float>;
        cudaError_t e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)V_SMEM);
        if (e != cudaSuccess) return e;
        kv<<<(unsigned)(2 * (int64_t)a.N * a.H), SCAN_THREADS, V_SMEM, stream>>>(a, hdr, rec, win);
        return cudaGetLastError();
    }
    // the output gate fused into the output store needs whole rows of V: one
    // CTA per (sequence, head)
    auto kern = a.out_norm ? (a.out_bf16 ? chunk_scan_kernel<__nv_bfloat16, true>
                                         : chunk_scan_kernel<float, true>)
                           : (a.out_bf16 ? chunk_scan_kernel<__nv_bfloat16, false>
                                         : chunk_scan_kernel<float, false>);
    const uint32_t smem = a.out_norm ? S_SMEM_NORM : S_SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)((int64_t)a.N * a.H), SCAN_THREADS, smem, stream>>>(a, hdr, rec, win);
    return cudaGetLastError();
}

// Overlap of preparation and scan, on the caller's stream alone.  The scan
// keeps one CTA per (sequence, head) busy for the whole call; when those CTAs
// leave most SMs idle (few long sequences), the chunks are cut into windows
// and the launches go prep(0), scan(0), prep(1), scan(1), ...  Each scan
// window lets the next preparation window start once all its CTAs are
// resident (programmatic dependent launch), so that preparation fills the SMs
// the scan leaves free; each scan is an ordinary launch, so it starts after
// the preparation of its window, and that preparation's last CTA waits for
// the previous scan.
constexpr int kWindowChunks = 32;              // at least this many chunks per window
constexpr int kLastWindowThirds = 1;          // the last window's scan runs alone: a third as long

// Window w covers the global chunks [window_bound(w), window_bound(w + 1)).
int64_t window_bound(int64_t chunks, int W, int w)
{
    if (w >= W) return chunks;
    // W - 1 windows of three thirds, the last of kLastWindowThirds
    return chunks * (3 * w) / (3 * (W - 1) + kLastWindowThirds);
}

// Scratch of the no-allocation entry point (kda_chunk_fwd_static): a
// file-scope device array, so that call allocates nothing.  Nothing in it has
// to start at zero: the plan kernel writes the whole header and the
// preparation writes every record the scan reads.
// Every GPU that loads the library holds these bytes until the process exits,
// and they keep the last call's contents.  In host code the name is only a
// host-side stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_static_scratch_ptr[kMaxDevices];
std::mutex g_static_scratch_mu;

}  // namespace

cudaError_t static_scratch(void** ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* p = g_static_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        // set-up, once per device, with that device current
        std::lock_guard<std::mutex> lock(g_static_scratch_mu);
        p = g_static_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            e = cudaGetSymbolAddress(&p, g_static_scratch);
            if (e != cudaSuccess) return e;
            g_static_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *ptr = p;
    return cudaSuccess;
}

int64_t chunk_plan_header_bytes(int32_t N) { return header_bytes(N); }

cudaError_t launch_chunk_plan(const int32_t* cu, int32_t N, int64_t T, int32_t* hdr,
                              int32_t* status, cudaStream_t stream)
{
    static_assert(kHdrOff == kPlanOffsets, "plan header layout");
    chunk_plan_kernel<<<1, 1024, 0, stream>>>(cu, N, T, hdr, status);
    return cudaGetLastError();
}


// Workspace: plan header, one record per chunk bound and head, then the
// windows' state carry [N,H,K,V] FP32.
int64_t split_workspace_bytes(int32_t N, int64_t T, int32_t H)
{
    return header_bytes(N) + split_chunk_bound(N, T) * H * (int64_t)REC_BYTES +
           (int64_t)N * H * DK * DV * 4;
}

cudaError_t launch_chunk_split(const ChunkArgs& a, int64_t chunks, bool overlap,
                               cudaStream_t stream)
{
    int32_t* hdr = static_cast<int32_t*>(a.workspace);
    unsigned char* rec = static_cast<unsigned char*>(a.workspace) + header_bytes(a.N);
    float* carry = reinterpret_cast<float*>(rec + split_chunk_bound(a.N, a.T) * a.H * (int64_t)REC_BYTES);
    const int64_t units = chunks * a.H;
    if (units > INT32_MAX || (int64_t)a.N * a.H > INT32_MAX) return cudaErrorInvalidConfiguration;
    PrepMaps maps;
    cudaError_t e = units > 0 ? make_prep_maps(a, &maps) : cudaSuccess;
    if (e != cudaSuccess) return e;
    chunk_plan_kernel<<<1, 1024, 0, stream>>>(a.cu_seqlens, a.N, a.T, hdr, a.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    const int sms = device_sm_count() > 0 ? device_sm_count() : 152;
    const int64_t heads = (int64_t)a.N * a.H;
    const int64_t W_shape = heads <= sms ? std::min<int64_t>(kMaxWindows, chunks / kWindowChunks) : 1;
    const int W = overlap ? (int)std::max<int64_t>(W_shape, 1) : 1;
    // The scan in V halves shortens the state's chain but streams the records
    // twice as fast and holds twice the SMs: it pays only for problems too
    // short for windows whose CTAs fit the GPU at once.  Windowed problems keep
    // the full-width scan (so that the preparation beside it keeps more SMs),
    // also when run in one window (kda_chunk_fwd_static): the choice depends on
    // the problem's shape alone, so both entry points give the same bits.
    const bool halves = !a.out_norm && W_shape <= 1 && 2 * heads <= sms;
    int32_t* ctr = window_counters(hdr, a.N);
    if (W <= 1) {
        e = launch_prep(a, maps, hdr, rec, 0, units, ctr, false, stream);
        if (e != cudaSuccess) return e;
        return launch_scan(a, hdr, rec, ScanWindow{0, INT32_MAX, nullptr, 1}, halves, stream);
    }
    for (int w = 0; w < W && e == cudaSuccess; ++w) {
        const int32_t g0 = (int32_t)window_bound(chunks, W, w);
        const int32_t g1 = (int32_t)window_bound(chunks, W, w + 1);
        e = launch_prep(a, maps, hdr, rec, (int64_t)g0 * a.H, (int64_t)(g1 - g0) * a.H, ctr + w,
                        w > 0, stream);
        const ScanWindow win{g0, w + 1 == W ? INT32_MAX : g1, carry, w + 1 == W ? 1 : 0};
        if (e == cudaSuccess) e = launch_scan(a, hdr, rec, win, halves, stream);
    }
    return e;
}

}  // namespace kda
