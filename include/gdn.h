/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta rule library, libgdn_gb300.so.
 *
 * The operation is the gated delta rule.  In the paper's orientation the state
 * S_t is d_v x d_k:
 *
 *     S_t = S_{t-1} ( alpha_t (I - beta_t k_t k_t^T) ) + beta_t v_t k_t^T,
 *     o_t = scale * S_t q_t
 *
 * Sources:
 *   - "TileLang 实战：KDA 从零到一 -- Gated DeltaNet", the opening equation
 *     and §2.3 (chunkwise algorithm, paper eqs 11-12).
 *   - "Gated Delta Network (GDN)", eq. 4 (the recurrence), eq. 12 (decode)
 *     and §4 (chunkwise training / prefill).
 *   - "You Could Have Come Up With Kimi Delta Attention", the KDA variant
 *     with a per-key-channel retention.
 *
 * Conventions shared by every entry point
 *   - Gates are natural logs: g = log alpha <= 0.  GDN has one gate per
 *     (token, head); KDA has one per (token, head, key channel).
 *   - beta is the writing strength.  The pages' range is (0, 1); (0, 2) is
 *     accepted as written, and no range check is made.
 *   - States use the transposed layout, like the pages' kernels:
 *     h = S^T, shape [N, H, d_k, d_v], fp32, row-major.  Row c is key
 *     channel c.
 *   - All tensors are contiguous row-major device buffers.  The caller
 *     allocates them and keeps ownership.  The library keeps no pointer
 *     after a call returns.
 *   - Each call is asynchronous on `stream`, a cudaStream_t (NULL means the
 *     legacy default stream).  A GDN_OK return means the work was enqueued.
 *     Kernel-side faults surface at the next synchronising CUDA call.
 *     Bounded waits that gave up are reported by gdn_device_status().
 *   - Arguments are checked on the host before any launch.  On an error
 *     nothing is launched, the status code says why, and gdn_last_error()
 *     holds a message (thread-local).
 *   - dtype is the element type of q, k and v (GDN_F32 or GDN_BF16); o_dtype
 *     is the element type of o (GDN_F32 or GDN_BF16; a bf16 output is the
 *     round-to-nearest-even of the fp32 result).  g, beta and the states are
 *     always fp32.
 *   - Buffers the call reads may not alias buffers it writes.  The one
 *     exception is gdn_recurrent_step's in-place state.
 *
 * Device memory is allocated only where an entry point says so: a chunk call
 * given no workspace allocates one on its stream and frees it there.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, inconsistent flags: nothing launched */
    GDN_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement: nothing launched */
    GDN_ERR_CUDA = 3,         /* a CUDA runtime call failed (device query, attribute, launch) */
    GDN_ERR_TIMEOUT = 4,      /* a kernel's bounded wait gave up (see gdn_device_status) */
    GDN_ERR_NONFINITE = 5     /* a chunk forward wrote a non-finite value (see gdn_device_status) */
} gdn_status;

typedef enum gdn_dtype {
    GDN_F32 = 0,   /* q, k, v, o are float */
    GDN_BF16 = 1   /* q, k, v, o are bfloat16 (round-to-nearest-even on output) */
} gdn_dtype;

/* Kernel choice for the chunk forward. */
typedef enum gdn_algo {
    GDN_ALGO_AUTO = 0,      /* the fastest tensor-core path that applies, else the generic one */
    GDN_ALGO_GENERIC = 1,   /* fp32 SIMT chunk kernel: any dtype, 1 <= d_k, d_v <= 256 where its fp32
                               tiles fit one CTA's shared memory (d_k = 256: chunk 64 for the
                               scalar gate, chunk <= 32 for the per-channel gate);
                               GDN_ERR_UNSUPPORTED otherwise */
    GDN_ALGO_TCGEN05 = 2,   /* retired (an earlier single-launch kernel, slower than the two-pass
                               path): always GDN_ERR_UNSUPPORTED */
    GDN_ALGO_TWO_PASS = 3   /* tcgen05 in two passes: a per-chunk kernel over all SMs writes the
                               state-independent products to a device workspace, then a state
                               kernel walks each chain.  bf16, chunk 64, d_k = d_v = 128, or
                               d_k = d_v = 256 with the scalar gate (its state kernel walks each
                               (chain, half of d_v)); GDN_ERR_UNSUPPORTED when the request does
                               not fit it.
                               Range: these kernels round some intermediates to fp16, whose
                               largest finite value is 65,504: the k and v values (scalar
                               gate), the per-chunk products P = scale (Gamma * Q K^T),
                               T diag(beta) and the corrections Delta = U - W S^T of every
                               chunk (per-channel gate also scale gamma Q, the decayed keys,
                               W, U and T).  With unit-norm q and k, beta in (0, 2) and |v|
                               up to about 1e3 they stay far inside it.  A value past it turns
                               into inf, and o or the final state then holds a non-finite
                               value: the state kernels check everything they write and
                               gdn_device_status reports GDN_ERR_NONFINITE. */
} gdn_algo;

/*
 * gdn_chunk_fwd -- chunkwise forward of the gated delta rule: training and
 * prefill, any sequence length.
 *
 * Sources: "TileLang 实战：KDA 从零到一 -- Gated DeltaNet", §2.3 (paper eqs
 * 11-12; the per-chunk triangular system and the UT transform), and
 * "Gated Delta Network (GDN)", §4(b3)-(d) (intra-chunk WY/UT products, then
 * the serial inter-chunk state pass).  The result is that of the token
 * recurrence above; only rounding depends on chunk_size.
 *
 *   q, k        [B, T, H, d_k]   dtype
 *   v           [B, T, H, d_v]   dtype
 *   g           [B, T, H]        fp32, log alpha (natural log)
 *   beta        [B, T, H]        fp32
 *   scale       output scale (commonly 1/sqrt(d_k))
 *   initial_state  [N, H, d_k, d_v] fp32, or NULL for zeros
 *   output_final_state  nonzero: write the state after each sequence's last token
 *   final_state [N, H, d_k, d_v] fp32; must be non-NULL iff output_final_state
 *   cu_seqlens  NULL: B independent sequences of T tokens (N = B).
 *               Otherwise int32 device array [n_seqs + 1] of packed sequence
 *               offsets: B must be 1, N = n_seqs >= 1, cu_seqlens[0] = 0,
 *               non-decreasing, cu_seqlens[n_seqs] = T.  Each sequence starts
 *               from its own initial state; chunks align to each sequence's
 *               start ("Gated Delta Network (GDN)", §6: chunk boundaries are
 *               not sequence boundaries).  Zero-length sequences are allowed
 *               (final = initial).  The contents are on the device and are not
 *               checked on the host.  The kernels clamp every offset into
 *               [0, T], so a malformed array cannot make them touch memory out
 *               of bounds, but the results are then unspecified.
 *   o           [B, T, H, d_v]   o_dtype (output)
 *   chunk_size  16, 32 or 64 (the pages' kernels use these; 64 is the default there)
 *   sizes       B >= 1, T >= 0, H >= 1, 1 <= d_k, d_v <= 256 (the pages' bound on
 *               the head sizes; the tensor-core path takes 128 and, for this scalar
 *               gate, 256; other sizes run on the generic kernel)
 *
 * Packed sequences give results bitwise equal to running each sequence alone.
 */
gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         float scale, const float* initial_state, int output_final_state, float* final_state,
                         const int32_t* cu_seqlens, int n_seqs, void* o,
                         int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype,
                         void* stream);

/* gdn_chunk_fwd with an explicit kernel choice (for tests and measurement). */
gdn_status gdn_chunk_fwd_algo(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              float scale, const float* initial_state, int output_final_state,
                              float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o,
                              int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                              gdn_dtype o_dtype, gdn_algo algo, void* stream);

/*
 * gdn_chunk_fwd_ws -- gdn_chunk_fwd with an explicit kernel choice and a
 * caller-provided device workspace for the kernels that need one
 * (GDN_ALGO_TWO_PASS; see gdn_chunk_workspace_size).
 *   workspace        device memory, 256-byte aligned, at least the size
 *                    gdn_chunk_workspace_size reports; owned by the caller and
 *                    used only by the work this call enqueues on `stream`, so
 *                    it may be reused once that work is ordered before the
 *                    reuse.  Two calls in flight at once must not share it.
 *                    NULL: the library allocates it on `stream` for the call
 *                    (stream-ordered allocation) and frees it after the work.
 *   workspace_bytes  its size; GDN_ERR_INVALID_ARG if too small.
 */
gdn_status gdn_chunk_fwd_ws(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            float scale, const float* initial_state, int output_final_state,
                            float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o,
                            int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                            gdn_dtype o_dtype, gdn_algo algo, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Optional in-kernel activation of the scalar gate and of beta ("Gated Delta
 * Network (GDN)", §3.1 eq. 5 gives the parameterisation; §4 and §6 describe
 * fusing it into the kernel so no separate activation pass runs):
 *   A_log         [H] fp32 device, or NULL: g already holds log alpha.  When set,
 *                 g holds raw logits x and the kernel uses
 *                 log alpha = -exp(A_log[h]) * softplus(x + dt_bias[h]).
 *   dt_bias       [H] fp32 device, or NULL (zero); needs A_log.
 *   beta_sigmoid  0: beta is used as given.  1: beta holds logits and the kernel
 *                 uses sigmoid(beta).  2: the kernel uses 2 sigmoid(beta), so beta
 *                 lies in (0, 2) and the transition I - beta k k^T of a unit key
 *                 may have a negative eigenvalue (the §5 implementation notes of
 *                 the same page).  Other values: GDN_ERR_INVALID_ARG.
 * The gate activation (A_log, dt_bias) applies to the scalar gate only; the
 * per-channel (KDA) entries accept beta_sigmoid alone.
 */
typedef struct gdn_gate_act {
    const float* A_log;
    const float* dt_bias;
    int beta_sigmoid;
} gdn_gate_act;

/*
 * gdn_chunk_fwd_act -- gdn_chunk_fwd_ws with the gate / beta activation in the
 * kernel (act may be NULL: no activation).  The activation runs on the
 * two-pass path only; another kernel choice returns GDN_ERR_UNSUPPORTED.
 */
gdn_status gdn_chunk_fwd_act(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             float scale, const float* initial_state, int output_final_state,
                             float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o,
                             int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                             gdn_dtype o_dtype, const gdn_gate_act* act, gdn_algo algo, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * gdn_chunk_fwd_ex -- the chunk forward with every option in one call:
 *   per_channel   nonzero: the KDA gate (g [B, T, H_v, d_k]), as kda_chunk_fwd.
 *   H_k, H_v      grouped value heads ("Gated Delta Network (GDN)", §4: more
 *                 value heads than key heads): q and k are [B, T, H_k, d_k];
 *                 v, o, g, beta and the states are per value head; value head
 *                 h uses key head h / (H_v / H_k).  H_v must be a multiple of
 *                 H_k (H_k = H_v is plain GDN).
 *   act           the gate / beta activation (may be NULL).
 * Grouped heads and the activation run on the two-pass path only; another
 * kernel choice returns GDN_ERR_UNSUPPORTED.  Other arguments are those of
 * gdn_chunk_fwd_ws.
 */
gdn_status gdn_chunk_fwd_ex(int per_channel, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float scale, const float* initial_state, int output_final_state,
                            float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o,
                            int B, int T, int H_k, int H_v, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                            gdn_dtype o_dtype, const gdn_gate_act* act, gdn_algo algo, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * kda_chunk_fwd -- chunkwise forward of Kimi Delta Attention.  The retention
 * is a per-key-channel vector exp(g_t), applied as Diag(exp g_t) on the key
 * side of the state before the delta update.
 *
 * Source: "You Could Have Come Up With Kimi Delta Attention": the recurrent
 * five-step update (decay, predict, residual, rank-1 write, read) and its
 * chunkwise form, with per-channel decays between tokens, the strictly lower
 * key-key system and the read matrix that includes the diagonal.
 *
 * Arguments and layouts are those of gdn_chunk_fwd, except that g is
 * [B, T, H, d_k] fp32.  With g equal on every channel the result is the GDN
 * result.
 */
gdn_status kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         float scale, const float* initial_state, int output_final_state, float* final_state,
                         const int32_t* cu_seqlens, int n_seqs, void* o,
                         int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype, gdn_dtype o_dtype,
                         void* stream);

gdn_status kda_chunk_fwd_algo(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              float scale, const float* initial_state, int output_final_state,
                              float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o,
                              int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                              gdn_dtype o_dtype, gdn_algo algo, void* stream);

/* kda_chunk_fwd with an explicit kernel choice and workspace, as gdn_chunk_fwd_ws. */
gdn_status kda_chunk_fwd_ws(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            float scale, const float* initial_state, int output_final_state,
                            float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o,
                            int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                            gdn_dtype o_dtype, gdn_algo algo, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * gdn_chunk_fwd_noalloc -- the two-pass chunk forward (GDN_ALGO_TWO_PASS;
 * per_channel nonzero: the KDA gate, as kda_chunk_fwd) with its workspace in a
 * statically allocated device array of the library instead of caller or
 * stream-ordered memory: the call allocates and frees nothing.  The pages
 * describe no counterpart; this entry point exists for callers that must not
 * allocate (for example inside a captured graph's replay loop).
 *   Limit: the static scratch holds 64 MiB: (floor(B*T / 64) + N + 1) * H
 *   records of gdn_chunk_workspace_size's per-item size (32,768 bytes for the
 *   scalar gate at d = 128, 114,688 at d = 256, 74,240 for the per-channel
 *   gate) must fit in 67,108,864 bytes: 2,048 scalar-gate items at d = 128
 *   (e.g. one 4096-token sequence with 31 heads), 585 at d = 256 (8 heads), or
 *   903 per-channel ones (13 heads).  A larger request returns
 *   GDN_ERR_UNSUPPORTED with the sizes in the message and launches nothing.
 *   Sharing: every call on a device uses the same scratch, so calls whose work
 *   can overlap (different streams, or threads without ordering) race and give
 *   unspecified results; order them on one stream.  Nothing in the scratch
 *   needs to start at zero: each call writes every byte it later reads.
 *   Set-up: the first call on a device looks the scratch up
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 * Other arguments, layouts and status codes are those of gdn_chunk_fwd.
 */
gdn_status gdn_chunk_fwd_noalloc(int per_channel, const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, float scale, const float* initial_state, int output_final_state,
                                 float* final_state, const int32_t* cu_seqlens, int n_seqs, void* o,
                                 int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                                 gdn_dtype o_dtype, void* stream);

/*
 * gdn_recurrent_step -- one decode token for N independent sequences.
 *
 * Sources: "Gated Delta Network (GDN)", eq. 12 and §4.4 (decode runs the
 * recurrent form, one token at a time, at a constant cost per token), and
 * the fused recurrent kernel on "You Could Have Come Up With Kimi Delta
 * Attention" (decay, predict, residual, rank-1 write, read).
 *
 *   q, k   [N, H, d_k] dtype      v  [N, H, d_v] dtype      o  [N, H, d_v] o_dtype
 *   g      [N, H] fp32 (log alpha)   beta [N, H] fp32
 *   state  [N, H, d_k, d_v] fp32, updated in place (the only aliasing allowed)
 *   o      output: o = scale * S_t q_t, read after the write
 *   sizes  N >= 1, H >= 1, 1 <= d_k, d_v <= 256
 */
gdn_status gdn_recurrent_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              float scale, float* state, void* o, int N, int H, int d_k, int d_v,
                              gdn_dtype dtype, gdn_dtype o_dtype, void* stream);

/* gdn_recurrent_step with the gate / beta activation of gdn_gate_act in the kernel (act may be NULL). */
gdn_status gdn_recurrent_step_act(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                  float scale, float* state, void* o, int N, int H, int d_k, int d_v,
                                  gdn_dtype dtype, gdn_dtype o_dtype, const gdn_gate_act* act, void* stream);

/*
 * gdn_recurrent_step_ex -- the decode step with every option: per_channel
 * (the KDA gate, g [N, H_v, d_k]), grouped value heads (q, k [N, H_k, d_k];
 * value head h uses key head h / (H_v / H_k)) and the activation (may be NULL).
 */
gdn_status gdn_recurrent_step_ex(int per_channel, const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, float scale, float* state, void* o, int N, int H_k, int H_v,
                                 int d_k, int d_v, gdn_dtype dtype, gdn_dtype o_dtype, const gdn_gate_act* act,
                                 void* stream);

/*
 * kda_recurrent_step -- one decode token of Kimi Delta Attention for N
 * independent sequences: the retention is the per-key-channel vector exp(g),
 * applied as Diag(exp g) on the key side of the state before the delta update.
 *
 * Source: "You Could Have Come Up With Kimi Delta Attention", the fused
 * recurrent form (decay per channel, predict, residual, rank-1 write, read).
 *
 * Arguments and layouts are those of gdn_recurrent_step, except that g is
 * [N, H, d_k] fp32.  With g equal on every channel the result is the GDN step.
 */
gdn_status kda_recurrent_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              float scale, float* state, void* o, int N, int H, int d_k, int d_v,
                              gdn_dtype dtype, gdn_dtype o_dtype, void* stream);

/*
 * gdn_chunk_plan -- which kernel a chunk-forward call with these sizes would run.
 * The buffers are assumed to be 16-byte aligned.  per_channel nonzero stands
 * for kda_chunk_fwd; varlen nonzero stands for a call with cu_seqlens.
 * requested is resolved into *chosen: GDN_ALGO_AUTO becomes
 * GDN_ALGO_TWO_PASS or GDN_ALGO_GENERIC.  The status is the one the call
 * itself would return for these sizes, and *chosen is written only on GDN_OK.
 * Nothing is launched.
 */
gdn_status gdn_chunk_plan(int per_channel, int B, int T, int H, int d_k, int d_v, int chunk_size,
                          gdn_dtype dtype, gdn_dtype o_dtype, int varlen, gdn_algo requested,
                          gdn_algo* chosen);

/*
 * gdn_chunk_workspace_size -- device workspace bytes of a chunk-forward call
 * with these sizes and kernel request (0 when the resolved kernel needs
 * none).  n_seqs is 0 for a call without cu_seqlens, else its number of
 * packed sequences.  The two-pass kernels keep a record per (chunk slot,
 * head): for the scalar gate at d = 128 32,768 bytes (-W, P^T and
 * T diag(beta) in fp16, with W = T diag(beta gamma) K); at d = 256 114,688
 * bytes (the same plus Q~ = diag(scale gamma) Q and K~ = diag(gamma_C/gamma) K
 * in fp16); for the per-channel gate 74,240 bytes ([Q^; W] with
 * Q^ = scale gamma Q, Ktilde, U and P in fp16, and gamma_C).
 * There are floor(B*T / 64) + N + 1 slots.  Same status rules as
 * gdn_chunk_plan.
 */
gdn_status gdn_chunk_workspace_size(int per_channel, int B, int T, int H, int d_k, int d_v, int chunk_size,
                                    gdn_dtype dtype, gdn_dtype o_dtype, int n_seqs, gdn_algo requested,
                                    size_t* bytes);

/*
 * gdn_chunk_bwd -- gradients of the chunk forward (gdn_chunk_fwd with
 * per_channel = 0, kda_chunk_fwd with per_channel = 1).  The pages give the
 * chunkwise backward of the ungated delta rule ("阅读笔记：DeltaNet 在 FLA 中的
 * 代码实现", 二、反向传播, steps 1-6); this call computes the same gradients for
 * the gated forms.  It computes the gradients of
 *     L = sum <grad_o, o> + sum <grad_final_state, final state>
 * with respect to q, k, v, g, beta and initial_state, where o and the final
 * state are those of the forward with the same inputs.  It takes the forward's
 * inputs, not its outputs: a first kernel recomputes the state entering every
 * chunk into the workspace, a second walks the chunks from the last to the
 * first.  All arithmetic is fp32.
 *   q, k, v, g, beta, scale, initial_state, cu_seqlens, n_seqs, B, T, H, d_k,
 *   d_v, dtype: as gdn_chunk_fwd / kda_chunk_fwd (g [B, T, H] or
 *   [B, T, H, d_k] by per_channel).
 *   grad_o            [B, T, H, d_v] device, of type do_dtype (GDN_F32 or GDN_BF16).
 *   grad_final_state  [N, H, d_k, d_v] fp32 device, or NULL (zero).
 *   grad_q, grad_k    [B, T, H, d_k] fp32 device, written.
 *   grad_v            [B, T, H, d_v] fp32 device, written.
 *   grad_g            fp32 device, the shape of g, written.
 *   grad_beta         [B, T, H] fp32 device, written.
 *   grad_initial_state  [N, H, d_k, d_v] fp32 device, or NULL (not written).
 *   chunk_size        16 or 32, or 0: the largest that fits one CTA's shared
 *                     memory.  It sets the granularity of the recomputation,
 *                     not the result (which is exact up to rounding).
 *   workspace         device memory for the chunk-entry states, 256-byte
 *                     aligned, at least gdn_chunk_bwd_workspace_size bytes;
 *                     NULL: allocated and freed on `stream` for the call.
 * Tokens of a packed sequence only see their own sequence, as in the forward.
 * Every output is written in full (rows of empty sequences have none).
 * Errors: GDN_ERR_INVALID_ARG for NULL or misaligned buffers, bad sizes or a
 * short workspace; GDN_ERR_UNSUPPORTED for head sizes above 256 or a
 * (chunk_size, d_k) pair whose shared memory does not fit one CTA; GDN_ERR_CUDA
 * if a launch fails.  Nothing is written unless the status is GDN_OK.
 */
gdn_status gdn_chunk_bwd(int per_channel, const void* q, const void* k, const void* v, const float* g,
                         const float* beta, float scale, const float* initial_state, const void* grad_o,
                         const float* grad_final_state, const int32_t* cu_seqlens, int n_seqs, float* grad_q,
                         float* grad_k, float* grad_v, float* grad_g, float* grad_beta, float* grad_initial_state,
                         int B, int T, int H, int d_k, int d_v, int chunk_size, gdn_dtype dtype,
                         gdn_dtype do_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_chunk_bwd_act -- gdn_chunk_bwd with the gate and beta activations of
 * gdn_gate_act in the path (act may be NULL: plain gdn_chunk_bwd).  g and beta
 * then hold raw logits, as for gdn_chunk_fwd_act; the forward's activations are
 * log alpha = -exp(A_log) softplus(g + dt_bias) ("Gated Delta Network (GDN)",
 * §3.1 eq. 5) and beta = sigmoid or 2 sigmoid of the logit.  grad_g and
 * grad_beta receive the gradients of those raw logits, and
 *   grad_A_log    [H] fp32 device, required when A_log is given: sum over every
 *                 token of the gradient of log alpha times log alpha;
 *   grad_dt_bias  [H] fp32 device or NULL (needs dt_bias): sum over every
 *                 token of grad_g.
 * The per-head sums are reduced in a fixed order (run-to-run identical).  The
 * gate activation applies to the scalar gate only (GDN_ERR_UNSUPPORTED with
 * per_channel); the beta activation to both.
 */
gdn_status gdn_chunk_bwd_act(int per_channel, const void* q, const void* k, const void* v, const float* g,
                             const float* beta, float scale, const float* initial_state, const void* grad_o,
                             const float* grad_final_state, const int32_t* cu_seqlens, int n_seqs, float* grad_q,
                             float* grad_k, float* grad_v, float* grad_g, float* grad_beta, float* grad_initial_state,
                             float* grad_A_log, float* grad_dt_bias, int B, int T, int H, int d_k, int d_v,
                             int chunk_size, gdn_dtype dtype, gdn_dtype do_dtype, const gdn_gate_act* act,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_chunk_bwd_ex -- the general backward: gdn_chunk_bwd_act plus grouped
 * value heads, as gdn_chunk_fwd_ex.  q, k and grad_q, grad_k are
 * [B, T, H_k, d_k]; v, g, beta, the states and their gradients have H_v value
 * heads (a multiple of H_k; H_k = 0 means H_v).  Value head h reads key head
 * h / (H_v / H_k), so grad_q and grad_k of a key head sum its value heads'
 * parts (in head order, run-to-run identical).  The workspace then also holds
 * those parts (gdn_chunk_bwd_workspace_size_ex).
 */
gdn_status gdn_chunk_bwd_ex(int per_channel, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, float scale, const float* initial_state, const void* grad_o,
                            const float* grad_final_state, const int32_t* cu_seqlens, int n_seqs, float* grad_q,
                            float* grad_k, float* grad_v, float* grad_g, float* grad_beta, float* grad_initial_state,
                            float* grad_A_log, float* grad_dt_bias, int B, int T, int H_k, int H_v, int d_k, int d_v,
                            int chunk_size, gdn_dtype dtype, gdn_dtype do_dtype, const gdn_gate_act* act,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_chunk_bwd_workspace_size -- bytes of the gdn_chunk_bwd (and
 * gdn_chunk_bwd_act) workspace.  Per (chunk slot, head): the entry state and
 * the exit-state gradient (fp32 [d_k, d_v] each), Delta, Y and Z (fp32
 * [C, d_v] each) and a record of the chunk's state-independent products; then
 * room for the activated log alpha and beta (fp32 [B, T, H] each).  A batch
 * has B * (ceil(T / C) + 1) slots, packed sequences floor(T / C) + 2 n_seqs
 * (C the chunk the call takes; chunk_size 0 as in gdn_chunk_bwd).  n_seqs is 0
 * for a call without cu_seqlens.  The _ex form takes the key heads H_k too: with
 * H_k < H_v the workspace adds the per-value-head grad_q and grad_k parts (fp32
 * [B, T, H_v, d_k] each).
 */
gdn_status gdn_chunk_bwd_workspace_size_ex(int per_channel, int B, int T, int H_k, int H_v, int d_k, int d_v,
                                           int chunk_size, int n_seqs, size_t* bytes);
gdn_status gdn_chunk_bwd_workspace_size(int per_channel, int B, int T, int H, int d_k, int d_v, int chunk_size,
                                        int n_seqs, size_t* bytes);

/*
 * gdn_test_inject -- arm a one-shot test of the bounded waits.
 * GDN_TEST_BWD_RECORD_STALL, for the calling thread's next gdn_chunk_bwd call: the state walks
 * leave out the bulk copy of their first chunk record, so the bounded wait for
 * it gives up (after 2 s), the walk records the failure in the device status
 * and leaves; gdn_device_status then returns GDN_ERR_TIMEOUT, and that call's
 * gradients are unspecified.  No copy is left in flight and the context stays
 * usable.  0 disarms.  GDN_ERR_INVALID_ARG for an unknown value.
 */
#define GDN_TEST_BWD_RECORD_STALL 1
/*
 * GDN_TEST_FWD_RECORD_STALL: the same for the calling thread's next chunk
 * forward on the two-pass path (either gate): the state kernels leave out the
 * copies of the first chunk record of every chain, so their bounded waits give
 * up, gdn_device_status reports GDN_ERR_TIMEOUT and that call's outputs are
 * unspecified.  Nothing is left in flight and the context stays usable.
 * GDN_TEST_FWD_ONE_STAGE: the next scalar-gate two-pass forward refills the
 * two-stage buffers of its state kernel (at d = 128 every one of them, at
 * d = 256 those of [-W; Q~]) only after the previous chunk's products have
 * completed (one chunk in flight instead of two).  This changes the timing
 * only: the result must be bitwise the same.
 */
#define GDN_TEST_FWD_RECORD_STALL 2
#define GDN_TEST_FWD_ONE_STAGE 3
gdn_status gdn_test_inject(int what);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* gdn_last_error(void);

/*
 * Device-side status of the kernels that use bounded waits (the tcgen05 paths
 * and the chunk backward's state walks) and of the chunk forward's output
 * check.  Synchronises the current device.  It returns GDN_OK;
 * GDN_ERR_TIMEOUT if any CTA gave up a bounded wait since the status was last
 * cleared (a CTA that gives up drops its work and its outputs are
 * unspecified); else GDN_ERR_NONFINITE if a two-pass chunk forward wrote a
 * non-finite value to o or the final state (an fp16 intermediate passed
 * 65,504, see GDN_ALGO_TWO_PASS, or an input was not finite).  With clear
 * nonzero, the status is reset.  GDN_ERR_CUDA if the query itself failed.
 */
gdn_status gdn_device_status(int clear);

/* Library version string. */
const char* gdn_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* GDN_GB300_H */
