// Blackwell (sm_103a) tensor-core primitives: tcgen05 MMA with operands in
// shared memory and accumulators in tensor memory (TMEM), mbarrier waits
// bounded in time, and the 128-byte-swizzled shared-memory tile layout the
// MMA descriptors describe.  Inline PTX only.
#pragma once

#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- layouts
//
// SW128 tile: rows of 128 bytes, 8-row atoms of 1024 bytes, the 16-byte chunk
// j of row r stored at chunk position j ^ (r % 8).  A matrix wider than 128
// bytes along its contiguous dimension is stored as consecutive "blocks" of
// 128-byte rows: block b holds bytes [128 b, 128 b + 128) of every row.
//   offset(row, byte) = (byte / 128) * rows * 128 + sw128(row, byte % 128)
// Every block must start 1024-byte aligned.
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t byte_in_row)
{
    return (row >> 3) * 1024u + (row & 7u) * 128u +
           ((((byte_in_row >> 4) ^ (row & 7u)) << 4) | (byte_in_row & 15u));
}

__device__ __forceinline__ uint32_t sw128_tile(uint32_t rows, uint32_t row, uint32_t byte)
{
    return (byte >> 7) * rows * 128u + sw128(row, byte & 127u);
}

// Shared-memory matrix descriptor, SWIZZLE_128B.
//   bits 0-13 start >> 4, 16-29 leading byte offset >> 4, 32-45 stride byte
//   offset >> 4, 46-47 version (1), 61-63 layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// K-major operand (rows = M or N index, K contiguous) of `rows` rows.  k-step
// `s` covers 32 bytes of K (16 BF16 or 8 TF32 elements).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, uint32_t rows, uint32_t s)
{
    const uint32_t start = base + (s >> 2) * rows * 128u + (s & 3u) * 32u;
    return desc_sw128(start, 16u, 1024u);
}

// MN-major BF16 operand whose MN extent is exactly 64 elements (one 128-byte
// row per K index): rows are K indices.  k-step `s` covers K rows 16 s .. 16 s + 15.
__device__ __forceinline__ uint64_t desc_mnmajor64(uint32_t base, uint32_t s)
{
    return desc_sw128(base + s * 2048u, 8192u, 1024u);
}

// MN-major 16-bit operand with an MN extent of 128 elements: two 64-element
// groups, each stored as K rows of 128 bytes; group 1 starts `group_bytes`
// after group 0.  k-step `s` covers K rows 16 s .. 16 s + 15.
__device__ __forceinline__ uint64_t desc_mnmajor128(uint32_t base, uint32_t group_bytes, uint32_t s)
{
    return desc_sw128(base + s * 2048u, group_bytes, 1024u);
}

// Byte offsets of k-step s within the operands above, for desc_advance.
__host__ __device__ constexpr uint32_t kmajor_off(uint32_t rows, uint32_t s)
{
    return (s >> 2) * rows * 128u + (s & 3u) * 32u;
}
__host__ __device__ constexpr uint32_t mnmajor_off(uint32_t s) { return s * 2048u; }

// The descriptor of the same operand `bytes` further on (a multiple of 16).
// The start field holds the shared-memory address >> 4 in its low 14 bits;
// every shared-memory address fits, so the sum never carries out of it.
// Issuing from descriptors computed once keeps the issuing thread's integer
// work per MMA to one addition.
__device__ __forceinline__ uint64_t desc_advance(uint64_t d, uint32_t bytes)
{
    return d + (bytes >> 4);
}

// Instruction descriptor (kind::f16 with F16 or BF16 operands, or kind::tf32), FP32 D.
//   bits 4-5 D format (1 = F32), 7-9 A format, 10-12 B format (0 = F16,
//   1 = BF16, 2 = TF32), 15/16 A/B major (0 = K, 1 = MN), 17-22 N >> 3, 24-28 M >> 4.
constexpr uint32_t kFmtF16 = 0, kFmtBF16 = 1, kFmtTF32 = 2;
__host__ __device__ constexpr uint32_t idesc(uint32_t fmt, uint32_t M, uint32_t N,
                                             bool a_mn = false, bool b_mn = false)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ---------------------------------------------------------------- MMA
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                         uint32_t acc)
{
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}

// kind::f16 with F16 operands uses the same instruction as BF16; the format
// lives in the instruction descriptor.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                        uint32_t acc)
{
    mma_bf16(d_tmem, a, b, id, acc);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                         uint32_t acc)
{
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}

// Arrives once on `mbar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void commit(uint64_t* mbar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(mbar))
        : "memory");
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the MMA.
__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* m, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* m, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(m)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Nanoseconds on the GPU's global timer.
__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// How long a bounded wait polls before it gives up.  Every wait in these
// kernels is for work of the same CTA (an MMA group, a bulk copy, the other
// warps of the CTA), which takes microseconds; a second means an arrival was
// lost, and the kernel then reports KDA_ERR_TIMEOUT and returns.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Polls between two reads of the timer, and the most reads of it per wait (a
// second bound on the loop that does not depend on the timer).
constexpr uint32_t kPollsPerCheck = 64;
constexpr uint32_t kMaxTimerChecks = 1u << 20;

// Waits for phase `parity` to complete; false after about `limit_ns`.  The
// first batch of polls reads no timer: ordinary waits end there, and the
// timer read stays off the kernels' critical paths.
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    for (uint32_t j = 0; j < kPollsPerCheck; ++j)
        if (mbar_try_wait(m, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < kMaxTimerChecks; ++i) {
        for (uint32_t j = 0; j < kPollsPerCheck; ++j)
            if (mbar_try_wait(m, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Arrives on `m` and adds `bytes` to the transaction count its phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* m, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)),
                 "r"(bytes)
                 : "memory");
}

// Plain arrival (count 1) on `m`.
__device__ __forceinline__ void mbar_arrive(uint64_t* m)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(m)) : "memory");
}

// Named barrier `id` over `nthreads` threads (whole warps).
// Programmatic dependent launch: a grid launched with programmatic stream
// serialisation may start once every CTA of the grid before it has signalled
// (or exited); grid_dependency_wait() returns once that grid has completed and
// its memory operations are visible (at once when launched without it).
__device__ __forceinline__ void launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// As named_sync; returns whether any participating thread passed `pred` true.
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n.reg .pred pi, po;\nsetp.ne.u32 pi, %1, 0;\n"
        "bar.red.or.pred po, %2, %3, pi;\nselp.u32 %0, 1, 0, po;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- bulk copy
// Global -> shared bulk copy through the async proxy (both addresses 16-byte
// aligned, `bytes` a multiple of 16); completes `bytes` transactions on `m`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* m)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(m))
        : "memory");
}

// TMA tile load (cp.async.bulk.tensor, no multicast) of the box at
// coordinates (x, y, z) of a 3-D tensor map into shared memory (128-byte
// aligned), completing the box's bytes as transactions on `m`.  `tmap` is the
// generic address of a __grid_constant__ CUtensorMap kernel parameter; the
// innermost coordinate x times the element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z,
                                            uint64_t* m)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(m))
        : "memory");
}

// Hint: bring `bytes` (multiple of 16, 16-byte-aligned address) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- cp.async
// 16-byte global -> shared copy that bypasses registers; `valid` false fills zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------- TMEM
// Executed by one whole warp; the TMEM address is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

// Warp-collective: thread t of warp w reads TMEM lane 32 (w % 4) + t,
// columns [col, col + 32) of `taddr` (taddr's lane field = 32 (w % 4)).
// Waits for the load before returning.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32])
{
    uint32_t* u = reinterpret_cast<uint32_t*>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]),
          "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
          "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]),
          "=r"(u[31])
        : "r"(taddr)
        : "memory");
}

// As tmem_ld32 for 16 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16])
{
    uint32_t* u = reinterpret_cast<uint32_t*>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr)
        : "memory");
}

// Two 32-column loads (e.g. two accumulators of the same lanes) under one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float (&ra)[32],
                                            float (&rb)[32])
{
    uint32_t* u = reinterpret_cast<uint32_t*>(ra);
    uint32_t* w = reinterpret_cast<uint32_t*>(rb);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]),
          "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
          "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]),
          "=r"(u[31]), "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]),
          "=r"(w[5]), "=r"(w[6]), "=r"(w[7]), "=r"(w[8]), "=r"(w[9]), "=r"(w[10]),
          "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]), "=r"(w[15]), "=r"(w[16]),
          "=r"(w[17]), "=r"(w[18]), "=r"(w[19]), "=r"(w[20]), "=r"(w[21]), "=r"(w[22]),
          "=r"(w[23]), "=r"(w[24]), "=r"(w[25]), "=r"(w[26]), "=r"(w[27]), "=r"(w[28]),
          "=r"(w[29]), "=r"(w[30]), "=r"(w[31])
        : "r"(ta), "r"(tb)
        : "memory");
}

// Three 16-column loads under one wait.
__device__ __forceinline__ void tmem_ld16x3(uint32_t t0, uint32_t t1, uint32_t t2,
                                            float (&r)[48])
{
    uint32_t* u = reinterpret_cast<uint32_t*>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%48];\n"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]),
          "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
          "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]),
          "=r"(u[31]), "=r"(u[32]), "=r"(u[33]), "=r"(u[34]), "=r"(u[35]), "=r"(u[36]),
          "=r"(u[37]), "=r"(u[38]), "=r"(u[39]), "=r"(u[40]), "=r"(u[41]), "=r"(u[42]),
          "=r"(u[43]), "=r"(u[44]), "=r"(u[45]), "=r"(u[46]), "=r"(u[47])
        : "r"(t0), "r"(t1), "r"(t2)
        : "memory");
}

// Warp-collective: zeroes TMEM lane 32 (w % 4) + t, columns [col, col + 32)
// of `taddr`, and waits for the store.
__device__ __forceinline__ void tmem_zero32(uint32_t taddr)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,"
        "%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};\n"
        "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
        "r"(0u)
        : "memory");
}

__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col)
{
    return base + (lane << 16) + col;
}

}  // namespace tc
}  // namespace kda
