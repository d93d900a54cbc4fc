/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library
 * (libkda_gb300.so).
 *
 * The method: the gated delta-rule recurrence of Kimi Delta Attention with a
 * per-channel log-space decay,
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = scale * S_t^T q_t,
 *
 * over packed variable-length sequences, computed in chunks of 64 tokens.
 * Page references are to XTuner's pull requests "Add opt-in FP32 KDA chunk
 * computation" (#2301) and "GLM-5.3-Flash F6.2: KDA correctness and FLA
 * sequence parallelism" (#2153).
 *
 * Conventions shared by every entry point
 *   - Every array argument is a DEVICE pointer unless its name ends in
 *     `_host`.  Arrays are dense, row-major, in the layout given per argument,
 *     owned by the caller, and must stay valid until the stream reaches the
 *     launched work.  The library allocates no device memory.  Its only
 *     mutable global state is the static scratch of kda_chunk_fwd_static
 *     (calls of that entry point share it; see there) and the process-wide
 *     test switch of kda_test_set_fault; calls of every other entry point on
 *     different streams are independent.
 *   - Every device pointer must be 16-byte aligned (KDA_ERR_ALIGNMENT).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  The library never synchronises.
 *   - Argument errors are detected on the host before anything is launched:
 *     the call returns a non-zero kda_status and launches nothing.  A CUDA
 *     launch failure returns KDA_ERR_CUDA.  Errors that only the device can
 *     see (offsets that contradict T when no host mirror of cu_seqlens is
 *     given) are written to `*status_dev` when it is non-NULL: the kernel
 *     stores the first error code there and skips the bad unit; read it after
 *     the stream has reached the work.  The library never traps.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size, bad enum, bad offsets    */
    KDA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. K != 128)       */
    KDA_ERR_ALIGNMENT = 3,     /* a device pointer is not 16-byte aligned          */
    KDA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed             */
    KDA_ERR_TIMEOUT = 5,       /* device: a bounded wait gave up (status word)     */
    KDA_ERR_DEVICE_ARG = 6,    /* device: offsets outside [0, T] (status word)     */
    KDA_ERR_TOO_LARGE = 7,     /* kda_chunk_fwd_static: over its static scratch    */
    KDA_ERR_RANGE = 8          /* device: a non-finite output value (status word)  */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

typedef enum {
    /* 16-bit tensor-core operands with FP32 accumulation and an FP32 state;
     * output rel-L2 error against the FP64 recurrence is held below 3e-3.
     * The operands are FP16, so v (and q and k when qk_l2norm = 0), and the
     * state and the chunk's intermediates built from them, must stay within
     * FP16's range, |x| < 65504.  Out-of-range values become infinities that
     * reach the output; every kernel of this mode checks the values it
     * stores (output rows and final states) and writes KDA_ERR_RANGE to
     * *status_dev when one is not finite, so an overflow is never silent
     * (inputs that hold NaN or infinity are reported the same way). */
    KDA_MODE_BF16_TC = 0,
    /* FP32-exact: output rel-L2 error below 1e-5 with F32 output.  This is
     * the counterpart of the pages' opt-in FP32 chunk intermediates ("Add
     * opt-in FP32 KDA chunk computation", section Change), without their
     * TF32 caveat.  Without a workspace every product is an IEEE FP32 fused
     * multiply-add on CUDA cores.  With one (two phases, see
     * kda_chunk_workspace_size) the chunk preparation is IEEE FP32 on CUDA
     * cores and the state scan's products run on the tensor cores with each
     * FP32 operand held as a pair of FP16 values scaled by a power of two
     * (about 22 significant bits; three MMAs with FP32 accumulation per
     * product), so it keeps FP32's range: no FP16 limit applies. */
    KDA_MODE_FP32_EXACT = 1
} kda_mode;

/*
 * kda_gate -- log-space decay and write strength from their pre-activations.
 *
 *   g[t,h,c]  = -exp(A_log[h]) * softplus(f[t,h,c] + dt_bias[h,c])
 *   beta[t,h] = 1 / (1 + exp(-b[t,h]))
 *
 * The decay is computed outside the chunk kernel with FP32 A_log/dt_bias and
 * beta is a sigmoid of its logits ("GLM-5.3-Flash F6.2: KDA correctness and
 * FLA sequence parallelism", fused-gate commit).
 *
 *   f       [T, H, K]  f_dtype (F32 or BF16)   gate pre-activation
 *   A_log   [H]        F32
 *   dt_bias [H, K]     F32
 *   b       [T, H]     b_dtype (F32 or BF16)   beta logits
 *   g_out   [T, H, K]  F32  (written)          every value < 0
 *   beta_out[T, H]     F32  (written)          every value in (0, 1)
 * Requires T >= 0, H >= 1, 1 <= K and K % 4 == 0.  T == 0 launches nothing and
 * accepts NULL tensor pointers.
 */
kda_status kda_gate(const void* f, int32_t f_dtype, const float* A_log, const float* dt_bias,
                    const void* b, int32_t b_dtype, int64_t T, int32_t H, int32_t K,
                    float* g_out, float* beta_out, kda_stream_t stream);

/*
 * kda_chunk_workspace_size -- bytes of device workspace that kda_chunk_fwd and
 * kda_chunk_fwd_gated use for a problem of N sequences, T tokens and H heads.
 *
 * With a workspace, KDA_MODE_BF16_TC runs in two phases: every (chunk, head)
 * is first prepared in parallel over the whole GPU (the chunk solve's
 * state-independent part: pair sums, (I + A_kk)^-1, W, U and the decay
 * factors) into the workspace, then one pass per (sequence, head) carries the
 * state through the chunks ("Add opt-in FP32 KDA chunk computation", section
 * Problem: the chunk solve and the carried state).  Without one it runs a
 * single pass per (sequence, head) that does all of a chunk's work in order.
 * KDA_MODE_FP32_EXACT splits the same way: with a workspace of at least
 * this size every (chunk, head) is prepared in parallel in IEEE FP32 on CUDA
 * cores (Q', K'', A_qk, the decay factors and W, U), then two CTAs per
 * (sequence, head), one per half of V, carry the FP32 state with the scan's
 * products on the tensor cores as scaled FP16 pairs (see KDA_MODE_FP32_EXACT).
 * It meets the same tolerance as the single-pass FP32 kernel; the two need
 * not agree bit for bit.
 *
 * When N * H is at most the GPU's SM count (the scan then leaves SMs idle)
 * and there are at least 64 chunks, the chunks are cut into min(3, chunks /
 * 32) windows, the last a third as long as the others, launched as prep(0),
 * scan(0), prep(1), scan(1), ... on the caller's stream,
 * each preparation after the first with programmatic dependent launch, so
 * that it runs on the SMs the scan before it leaves free.  Results are bit
 * for bit those of one window.
 *
 * The size is a bound that holds for every cu_seqlens with these N and T:
 * a 1 KiB-aligned header of 2 N + 8 int32, then for KDA_MODE_BF16_TC
 * (T / 64 + N) * H records of 74240 bytes and N * H * K * V FP32 (the state
 * carried between windows), for KDA_MODE_FP32_EXACT (T / 64 + N) * H records
 * of 148224 bytes.
 * Arguments as kda_chunk_fwd; *bytes_host is host memory.
 */
kda_status kda_chunk_workspace_size(int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                                    int32_t mode, int64_t* bytes_host);

/*
 * kda_chunk_fwd -- chunked KDA forward over packed sequences.
 *
 * Sequence n covers rows cu_seqlens[n] .. cu_seqlens[n+1]-1 of every tensor
 * ("packed offsets": "Add opt-in FP32 KDA chunk computation", section
 * Change).  Each sequence starts from a zero state; chunks of 64 tokens start
 * at the sequence start, the last one possibly shorter.
 *
 *   q, k       [T, H, K]  qkv_dtype (F32 or BF16)
 *   v          [T, H, V]  qkv_dtype
 *   g          [T, H, K]  F32   log-space decay, must be <= 0 (kda_gate's output)
 *   beta       [T, H]     F32   write strength in [0, 1]
 *   cu_seqlens [N+1]      int32 device copy of the offsets, cu[0] = 0, cu[N] = T,
 *                                non-decreasing
 *   cu_seqlens_host [N+1] int32 HOST mirror of the same offsets, or NULL.  When
 *                                given it is validated on the host (bad offsets
 *                                -> KDA_ERR_INVALID_ARG, nothing launched);
 *                                when NULL the kernel checks each sequence's
 *                                range against [0, T] and reports
 *                                KDA_ERR_DEVICE_ARG through status_dev.
 *   N >= 0 sequences, T >= 0 tokens, H >= 1 heads, K = V = 128 (else
 *   KDA_ERR_UNSUPPORTED).
 *   scale      output scale (typically 1/sqrt(K)).
 *   qk_l2norm  1: q and k are L2-normalised per (token, head) inside the op,
 *              x / sqrt(sum x^2 + 1e-6) in FP32 ("Add opt-in FP32 KDA chunk
 *              computation", section Change); 0: used as given.
 *   mode       kda_mode.
 *   out        [T, H, V]  out_dtype (F32 or BF16), written for every covered row.
 *   initial_state [N, H, K, V] F32, or NULL (every sequence starts from zero):
 *              the state each sequence starts from (the pages' wrapper lacks
 *              one: "Add opt-in FP32 KDA chunk computation", section Change).
 *   final_state [N, H, K, V] F32, or NULL: the state after each sequence's
 *              last token (the initial state for an empty sequence).
 *              final_state may alias initial_state.
 *   workspace  device scratch of workspace_bytes bytes, or NULL (see
 *              kda_chunk_workspace_size).  KDA_MODE_BF16_TC with a workspace
 *              needs workspace_bytes >= kda_chunk_workspace_size(...) (else
 *              KDA_ERR_INVALID_ARG); its contents are overwritten and mean
 *              nothing after the call.  Calls that share one workspace must be
 *              ordered (same stream, or synchronised): the library does not
 *              guard it.  KDA_MODE_FP32_EXACT runs in two phases when
 *              workspace_bytes >= kda_chunk_workspace_size(...) for that mode
 *              (16-byte aligned, else KDA_ERR_ALIGNMENT) and in its single-pass
 *              kernel otherwise (a smaller workspace is not used).
 *   status_dev one device int32 or NULL; the kernel writes a kda_status there
 *              only on a device-detected error (the caller zeroes it).
 */
kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                         const float* g, const float* beta,
                         const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                         int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                         float scale, int32_t qk_l2norm, int32_t mode,
                         void* out, int32_t out_dtype, const float* initial_state,
                         float* final_state, void* workspace, int64_t workspace_bytes,
                         int32_t* status_dev, kda_stream_t stream);

/*
 * kda_chunk_fwd_gated -- kda_chunk_fwd with the gate fused into its prologue.
 *
 * Takes the gate's inputs instead of g and beta and forms, per element,
 *   g = -exp(A_log[h]) * softplus(f + dt_bias[h,c]),  beta = sigmoid(b)
 * without writing g or beta to memory.  KDA_MODE_FP32_EXACT uses kda_gate's
 * FP32 arithmetic, so its result equals kda_gate followed by kda_chunk_fwd
 * bit for bit.  KDA_MODE_BF16_TC needs only e^g, which it forms directly as
 * (1 + e^(f + dt_bias))^(-exp(A_log)) with the hardware exp2/log2
 * approximations (relative error below 1e-5, against the 2^-11 rounding of
 * its FP16 operands), so its result agrees with kda_gate + kda_chunk_fwd
 * within the mode's tolerance but not bit for bit.
 * The pages compute the gate outside the chunk kernel ("GLM-5.3-
 * Flash F6.2: KDA correctness and FLA sequence parallelism", fused-gate
 * commit, with FP32 A_log/dt_bias); fusing it here removes that launch and
 * its round trip of g, and with f in BF16 (the activation dtype of the gate
 * projection that produces it) the call reads 256 bytes of f per token and
 * head instead of the 512 bytes of an FP32 g.
 *
 *   f       [T, H, K]  F32 or BF16 (f_dtype)
 *   A_log   [H] F32, dt_bias [H, K] F32
 *   b       [T, H]     F32 or BF16 (b_dtype)
 * Every other argument as kda_chunk_fwd.
 */
kda_status kda_chunk_fwd_gated(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                               const void* f, int32_t f_dtype, const float* A_log,
                               const float* dt_bias, const void* b, int32_t b_dtype,
                               const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                               int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                               float scale, int32_t qk_l2norm, int32_t mode,
                               void* out, int32_t out_dtype, const float* initial_state,
                               float* final_state, void* workspace, int64_t workspace_bytes,
                               int32_t* status_dev, kda_stream_t stream);

/*
 * kda_chunk_fwd_gated_norm -- kda_chunk_fwd_gated followed by the output gate
 * with gated RMSNorm (kda_gated_rmsnorm), in one call:
 *
 *   out[t, h, v] = o[t, h, v] / sqrt(mean_v' o[t, h, v']^2 + eps) * weight[v]
 *                  * sigmoid(z[t, h, v])
 *
 * where o is kda_chunk_fwd_gated's output.  The pages name the low-rank output
 * gate (g_a_proj -> g_b_proj) and the gated-norm wrapper that follow the core
 * ("GLM-5.3-Flash F6.2: KDA correctness and FLA sequence parallelism", module
 * and FLA-SP commits).  In KDA_MODE_BF16_TC with a workspace and BF16 z the
 * gate is applied in the state scan's output store: each chunk's o rows are
 * normalised from their FP32 values in registers and never reach memory, so
 * the call reads z once and writes the gated output once instead of writing
 * o, reading it back and writing y.  Any other mode, workspace choice or z
 * dtype runs kda_chunk_fwd_gated into `out` and then kda_gated_rmsnorm on it
 * in place (two launches, the same result up to the rounding of o to
 * out_dtype).
 *
 *   z       [T, H, V]  F32 or BF16 (z_dtype)   output-gate pre-activation; must
 *                                              not be `out`
 *   weight  [V]        F32                     per-channel weight shared by heads
 *   eps     >= 0
 *   out     [T, H, V]  out_dtype               the gated output
 * Every other argument as kda_chunk_fwd_gated.  In KDA_MODE_BF16_TC a
 * non-finite stored value sets KDA_ERR_RANGE as for kda_chunk_fwd.
 */
kda_status kda_chunk_fwd_gated_norm(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                                    const void* f, int32_t f_dtype, const float* A_log,
                                    const float* dt_bias, const void* b, int32_t b_dtype,
                                    const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                    int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                                    float scale, int32_t qk_l2norm, int32_t mode,
                                    const void* z, int32_t z_dtype, const float* weight,
                                    float eps, void* out, int32_t out_dtype,
                                    const float* initial_state, float* final_state,
                                    void* workspace, int64_t workspace_bytes,
                                    int32_t* status_dev, kda_stream_t stream);

/*
 * kda_chunk_fwd_static -- kda_chunk_fwd in KDA_MODE_BF16_TC, two-phase, with
 * the library's own scratch instead of a caller workspace.  The pages have no
 * counterpart: this is an interface for callers that cannot allocate device
 * memory per call -- a process whose device-memory budget is fixed up front
 * (e.g. a server that has handed the rest of HBM to its caches), or C code
 * with no allocator of its own, for which a cudaMalloc/cudaFree pair per call
 * would also synchronise the device.
 *
 * The scratch is one file-scope device array of 64 MiB in the library, so
 * the call allocates nothing; every GPU that loads the library holds those
 * 64 MiB until the process exits, and they keep the last call's contents.
 * A problem whose kda_chunk_workspace_size(...) exceeds 64 MiB is rejected
 * with KDA_ERR_TOO_LARGE before anything is launched.  That bound counts
 * (T / 64 + N) * H records of 74240 bytes plus N * H * 64 KiB of state
 * carry, so for H = 64 and N = 1, T / 64 + N may be at most 13 (T <= 768
 * tokens), and every further sequence costs one more record per head and
 * 4 MiB of carry.
 * The first call on a device does set-up (it looks up the array's device
 * address, which may load the library's device code), so make it before any
 * stream capture.  The address is remembered per device for the life of the
 * process: after cudaDeviceReset (or any reset of the primary context) the
 * remembered address is stale and this entry point must not be called
 * again in that process.  `stream` must belong to the current device
 * (KDA_ERR_INVALID_ARG otherwise).  Every call on a device uses the same
 * scratch: calls that
 * overlap in time (on different streams, or from different host threads
 * without ordering) race on it and give undefined results.  Nothing in the
 * scratch needs to start at zero.  The result equals kda_chunk_fwd with mode
 * KDA_MODE_BF16_TC and a workspace, bit for bit.  Arguments as kda_chunk_fwd.
 */
kda_status kda_chunk_fwd_static(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                                const float* g, const float* beta,
                                const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                                float scale, int32_t qk_l2norm, void* out, int32_t out_dtype,
                                const float* initial_state, float* final_state,
                                int32_t* status_dev, kda_stream_t stream);

/*
 * kda_recurrent_step -- one token of the recurrence for each of N sequences
 * (the decode step: the pages' serving path runs the FP32 recurrence token by
 * token, "Add opt-in FP32 KDA chunk computation", section Problem).
 *
 *   q, k  [N, H, K], v [N, H, V]  qkv_dtype (F32 or BF16): token n of sequence n
 *   g     [N, H, K] F32 log-decay (<= 0), beta [N, H] F32
 *   state [N, H, K, V] F32, read and overwritten in place:
 *           S <- (I - beta k^ k^^T) Diag(e^g) S + beta k^ v^T
 *   out   [N, H, V] out_dtype: scale * S^T q^ with the updated S
 * IEEE FP32 arithmetic; q and k are L2-normalised when qk_l2norm = 1.
 * K = V = 128 (else KDA_ERR_UNSUPPORTED).  N = 0 launches nothing.
 */
kda_status kda_recurrent_step(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                              const float* g, const float* beta, int32_t N, int32_t H,
                              int32_t K, int32_t V, float scale, int32_t qk_l2norm,
                              float* state, void* out, int32_t out_dtype,
                              kda_stream_t stream);

/*
 * kda_gated_rmsnorm -- the output gate with gated RMSNorm applied to the
 * attention output, per (token, head) row of V values:
 *
 *   y[r, v] = o[r, v] / sqrt(mean_v' o[r, v']^2 + eps) * weight[v] * sigmoid(z[r, v])
 *
 * The pages name the low-rank output gate (g_a_proj -> g_b_proj) and the
 * "gated-norm" wrapper of the KDA module without printing a formula ("GLM-5.3-
 * Flash F6.2: KDA correctness and FLA sequence parallelism", module and FLA-SP
 * commits); this is the plain reading of them.
 *
 *   o      [rows, V]  o_dtype (F32 or BF16)   attention output, rows = T * H
 *   z      [rows, V]  z_dtype (F32 or BF16)   output-gate pre-activation
 *   weight [V]        F32                     per-channel weight, shared by heads
 *   eps    >= 0
 *   y      [rows, V]  y_dtype (F32 or BF16)   may alias o when y_dtype == o_dtype
 * FP32 arithmetic.  V = 128 (else KDA_ERR_UNSUPPORTED); rows = 0 launches
 * nothing and accepts NULL pointers.
 */
kda_status kda_gated_rmsnorm(const void* o, int32_t o_dtype, const void* z, int32_t z_dtype,
                             const float* weight, int64_t rows, int32_t V, float eps, void* y,
                             int32_t y_dtype, kda_stream_t stream);

/*
 * kda_chunk_bwd_workspace_size -- bytes of device scratch kda_chunk_bwd needs
 * for N sequences of T packed tokens and H heads (K = V = 128, else
 * KDA_ERR_UNSUPPORTED): the plan header, K x V FP32 states for the
 * checkpoints at every 16-token segment start (4 (T / 64 + N) per head, a
 * bound over every cu_seqlens), three FP32 copies of [T,H,K] x 3 + [T,H]
 * (the partial row sums of three of the four 32-column slices each head is
 * split into) and 16 state slices (K x 32 FP32) per persistent CTA, at most
 * 1024 CTAs (the states inside the segment being walked backwards).
 */
kda_status kda_chunk_bwd_workspace_size(int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                                        int64_t* bytes_host);

/*
 * kda_chunk_bwd -- the vector-Jacobian product of kda_chunk_fwd: given dout,
 * the gradient of a scalar loss with respect to every output row, and
 * dfinal_state, with respect to every final state, returns the gradients with
 * respect to q, k, v, g, beta and the initial state.  The pages check the
 * chunked backward against FP64 budgets ("Add opt-in FP32 KDA chunk
 * computation", section Validation) and print no formula; this is the chain
 * rule applied by hand to the token recurrence the forward computes,
 *   S'_t = Diag(e^{g_t}) S_{t-1},  d_t = beta_t (v_t - S'_t^T k^_t),
 *   S_t = S'_t + k^_t d_t^T,        o_t = scale S_t^T q^_t,
 * tokens walked backwards per (sequence, head), and then through the L2
 * normalisation q^ = q / sqrt(|q|^2 + 1e-6) (k alike) when qk_l2norm = 1.
 *
 * Inputs are those of kda_chunk_fwd (q, k, v [T,H,K|V] qkv_dtype; g [T,H,K]
 * and beta [T,H] F32; cu_seqlens device, cu_seqlens_host optional host copy
 * checked as there; initial_state [N,H,K,V] F32 or NULL for zeros), plus
 *   dout           [T,H,V]   dout_dtype (F32 or BF16)
 *   dfinal_state   [N,H,K,V] F32 or NULL (zeros)
 * Outputs, all F32 and written in full (every token of every sequence):
 *   dq, dk [T,H,K], dv [T,H,V], dg [T,H,K], dbeta [T,H];
 *   dinitial_state [N,H,K,V] or NULL (not computed).
 * No output may alias an input or another output (the same base pointer is
 * rejected with KDA_ERR_INVALID_ARG).  workspace: device, 16-byte aligned, at least
 * kda_chunk_bwd_workspace_size bytes, owned by the caller, contents on entry
 * irrelevant; calls sharing one workspace must be ordered on one stream.
 * FP32 arithmetic throughout: the forward is recomputed token by token from
 * checkpoints of the state every 16 tokens, so the gradients are those of the
 * exact recurrence (either forward mode's output approximates it).
 * Errors as kda_chunk_fwd; offsets outside [0, T] seen on the device set
 * KDA_ERR_DEVICE_ARG in status_dev and leave those sequences' outputs unwritten.
 */
kda_status kda_chunk_bwd(const void* q, const void* k, const void* v, int32_t qkv_dtype,
                         const float* g, const float* beta,
                         const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                         int32_t N, int64_t T, int32_t H, int32_t K, int32_t V,
                         float scale, int32_t qk_l2norm,
                         const void* dout, int32_t dout_dtype,
                         const float* initial_state, const float* dfinal_state,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta,
                         float* dinitial_state, void* workspace, int64_t workspace_bytes,
                         int32_t* status_dev, kda_stream_t stream);

/*
 * kda_test_set_fault -- TEST HOOK, not for production use (no page
 * counterpart).  Lets a test make a bounded device wait run out without
 * faulting the GPU: while it is set, CTA 0 of every launch of the named
 * kernel withholds one mbarrier arrival, its wait gives up after about one
 * second, the kernel writes KDA_ERR_TIMEOUT to *status_dev, lets its copies
 * and MMAs in flight finish, releases its tensor memory and returns; the
 * results of that launch are undefined.
 *   where = KDA_TEST_FAULT_NONE (0)         off (the default)
 *           KDA_TEST_FAULT_SCAN (1)         state scan of the two-phase path
 *                                           (an epilogue arrival is withheld)
 *           KDA_TEST_FAULT_PREP (2)         chunk preparation of the two-phase
 *                                           path (its first MMA group and the
 *                                           commit that signals it are withheld)
 *           KDA_TEST_FAULT_SINGLE_PASS (3)  the single-pass kernel (likewise)
 * The setting is process-wide and read at each launch; other values return
 * KDA_ERR_INVALID_ARG.
 */
#define KDA_TEST_FAULT_NONE 0
#define KDA_TEST_FAULT_SCAN 1
#define KDA_TEST_FAULT_PREP 2
#define KDA_TEST_FAULT_SINGLE_PASS 3
kda_status kda_test_set_fault(int32_t where);

/* Static text for a kda_status value ("unknown status" otherwise). */
const char* kda_status_string(int32_t status);

/* ABI revision of this header; bumped on any incompatible change (2: initial
 * state argument of kda_chunk_fwd; kda_chunk_fwd_gated; kda_recurrent_step.
 * 3: workspace arguments; kda_chunk_workspace_size.  Later additions that
 * change no existing signature keep the number: kda_chunk_fwd_static,
 * kda_gated_rmsnorm, kda_chunk_bwd_workspace_size, kda_chunk_bwd,
 * KDA_ERR_RANGE, kda_test_set_fault, kda_chunk_fwd_gated_norm). */
int32_t kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
