/*
 * kda.h -- C ABI of libkda, a GB300 (sm_103a) implementation of the Kimi
 * Delta Attention (KDA) operator.
 *
 * Operation (from "Kimi K3：从三条信息流到完整系统", wineandchord.com):
 *   §KDA 是带逐通道遗忘的 delta rule, eq. (1), per sequence and head:
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *       o_t = scale * S_t^T q_t
 *     S is dk x dv; Diag(alpha_t) scales the key-channel rows of S; o_t reads
 *     the state after token t's own write.
 *   §下界 log-decay 是一个 kernel 设计, eq. (5):
 *       g_t = g_min * Sigmoid(e^A * z_t),  alpha_t = e^{g_t},  g_min = -5
 *     where z_t (per key channel) is the caller's gate pre-activation g_raw.
 *   §从投影到 Chunkwise 的完整接口, eqs. (3)-(4): the chunkwise form that the
 *     prefill kernels evaluate (16-token tiles, exact in real arithmetic).
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers owned by the caller; the
 *     library allocates no device or host memory and keeps no pointer after
 *     the call returns (kda_chunk_fwd_split takes a caller workspace;
 *     kda_chunk_fwd_split_noalloc uses a fixed buffer inside the library).
 *   - Every call is asynchronous on the given stream (0 = legacy default
 *     stream).  A KDA_OK return means the work was validated and enqueued.
 *   - Tensors are dense and row-major ("contiguous") in the stated shape.
 *   - Alignment (KDA_ERR_ALIGN otherwise): q, k, v, g_raw, out and the
 *     state tensors 16 bytes (they are moved by TMA / vector loads); beta,
 *     A_log and a per-head (scalar) g_raw to their element size; cu_seqlens
 *     and accepted to 4 bytes.
 *   - Arguments are validated on the host before any launch; a rejected
 *     call enqueues nothing and leaves every output untouched.  No call
 *     aborts, traps on the device or throws across this boundary.
 *   - Outputs must not alias inputs, except decode's state (in place).
 *   - Head dimensions dk, dv must each be 32, 64 or 128.
 *   - The query scale defaults to 1 (the pages apply none).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stream handle: a cudaStream_t passes through unchanged. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_ARG = 1,     /* NULL required pointer, negative size, bad N/B   */
    KDA_ERR_DTYPE = 2,   /* unknown kda_dtype                                */
    KDA_ERR_SHAPE = 3,   /* unsupported dk/dv                                */
    KDA_ERR_ALIGN = 4,   /* pointer not 16-byte aligned                      */
    KDA_ERR_LAUNCH = 5,  /* CUDA rejected the launch (see kda_last_cuda_error) */
    KDA_ERR_TIMEOUT = 6, /* reserved: a bounded device wait gave up          */
    KDA_ERR_SCRATCH = 7  /* kda_chunk_fwd_split_noalloc: the call needs more
                            than KDA_SPLIT_SCRATCH_BYTES of scratch          */
} kda_status;

typedef enum {
    KDA_F32 = 0,         /* q, k, v, g_raw, beta, out in fp32                 */
    KDA_BF16 = 1         /* q, k, v, g_raw, beta, out in bf16                 */
} kda_dtype;

/*
 * Gate variants: how g_raw becomes the log-decay g (alpha = e^g).  The
 * update rules before KDA and the gate it replaced ("Kimi K3: Two point
 * eight trillion parameters, open weights, and forty-seven pages of how",
 * §What changed between the paper and the model).
 */
typedef enum {
    KDA_GATE_BOUNDED = 0,      /* eq. (5): g = g_min * Sigmoid(e^A z)             */
    KDA_GATE_LOG_DECAY = 1,    /* g_raw is g itself (expected <= 0)              */
    KDA_GATE_NEG_SOFTPLUS = 2, /* Kimi Linear: g = -Softplus(e^A z), unbounded   */
    KDA_GATE_NONE = 3          /* alpha = 1: the plain delta rule; g_raw unused  */
} kda_gate_mode;

/*
 * Optional parameters.  A zero-initialised struct (or a NULL pointer)
 * selects the pages' defaults.
 *   g_min : floor of the log-decay in eq. (5); 0 selects -5.
 *   A_log : DEVICE pointer to H fp32 values, the per-head log-scale A of
 *           eq. (5) (the logit is multiplied by e^A); NULL selects A = 0.
 *   scale : factor applied to o_t; 0 selects 1.
 *   gate_mode : a kda_gate_mode; 0 selects eq. (5).
 *   gate_per_head : 0 = one gate per key channel (KDA, g_raw [.., H, dk]);
 *           1 = one gate per token and head shared by every key channel
 *           (gated delta, g_raw [.., H]).
 * Every gate runs on the tensor-core prefill for bf16 with dk = dv = 128
 * and on the fp32 prefill otherwise.  Under the unbounded modes (LOG_DECAY,
 * NEG_SOFTPLUS), a 16-token tile whose cumulative decay would take e^{-b}
 * past fp32's range computes its in-tile products with one exponential per
 * position pair instead of dividing by the cumulative decay (the fp32
 * prefill always does so under these modes).
 */
typedef struct {
    float g_min;
    const float *A_log;
    float scale;
    int gate_mode;
    int gate_per_head;
} kda_params;

/*
 * kda_chunk_fwd -- prefill / forward over whole sequences.
 *
 * Inputs (dtype dt unless stated):
 *   q, k   [B, T, H, dk]   queries and keys, used as given (already
 *                          normalised by the caller's projection chain).
 *   v      [B, T, H, dv]   values.
 *   g_raw  [B, T, H, dk]   gate pre-activation z of eq. (5) ([B, T, H] with
 *                          gate_per_head; may be NULL with KDA_GATE_NONE).
 *   beta   [B, T, H]       write strength, already in (0, 1).
 *   init_state [N, H, dk, dv] fp32, or NULL for zeros: the state entering
 *                          each sequence (row = key channel).
 *   cu_seqlens [N + 1] int32 DEVICE array, or NULL.
 *          NULL : the B rows are N = B independent sequences of length T.
 *          set  : B must be 1; the T tokens are N packed sequences, sequence
 *                 n spanning tokens [cu_seqlens[n], cu_seqlens[n+1]).  The
 *                 array must start at 0, be non-decreasing and end at T.
 *                 The kernels clamp each span into [0, T], so a malformed
 *                 array yields unspecified values but never an
 *                 out-of-bounds access.  Empty sequences are allowed: their
 *                 final state equals their initial state.
 *   N      number of sequences (must equal B when cu_seqlens is NULL).
 * Outputs:
 *   out    [B, T, H, dv]   o_t for every token (dtype dt); required if B*T > 0.
 *   final_state [N, H, dk, dv] fp32, or NULL: the state after each
 *          sequence's last token.
 * Numerics: fp32 state, gates and accumulation.  On the bf16 path the
 * tensor-core operands are fp16 (an fp16 copy of the state, the residual and
 * the decay-scaled q, k; all bounded well inside fp16's range), tf32 for the
 * in-tile products whose factors span e^{+-80}, and exact bf16 parts for
 * T Diag(beta) V; the fp32 path computes in fp32 throughout.
 */
kda_status kda_chunk_fwd(kda_dtype dt, int B, int T, int H, int dk, int dv,
                         const void *q, const void *k, const void *v,
                         const void *g_raw, const void *beta,
                         const float *init_state,
                         const int32_t *cu_seqlens, int N,
                         void *out, float *final_state,
                         const kda_params *p, kda_stream_t stream);

/*
 * kda_chunk_fwd_checkpointed -- kda_chunk_fwd that also saves the state at
 * chosen positions inside each sequence, for a prefix cache that restores
 * from a boundary rather than from the start ("Kimi K3：从三条信息流到完整系统",
 * §在线推理：两类记忆必须共同命中, "hybrid prefix cache"; the checkpoint is the
 * same S_t that eq. (1) carries, so a later call resumed from it via
 * init_state continues the sequence).
 *
 * checkpoint_every: E > 0, a multiple of 16.  Sequence n of length L_n
 *   gets floor(L_n / E) checkpoints: checkpoint i (0-based) is the state
 *   after its first (i + 1) * E tokens (the last one equals final_state
 *   when E divides L_n).
 * checkpoints: DEVICE fp32 [checkpoint_rows, H, dk, dv], caller-owned,
 *   16-byte aligned.  Sequence n's checkpoints are rows r_n .. r_n +
 *   floor(L_n / E) - 1, r_n = sum over m < n of floor(L_m / E) (without
 *   cu_seqlens: r_n = n * floor(T / E)).  Rows at or past checkpoint_rows
 *   are never written; kda_checkpoint_rows gives the count to allocate.
 * checkpoints == NULL (or checkpoint_rows == 0) is kda_chunk_fwd itself.
 * Other arguments and errors as kda_chunk_fwd; KDA_ERR_ARG also for E not
 * a positive multiple of 16 or checkpoint_rows < 0 with a buffer given.
 */
kda_status kda_chunk_fwd_checkpointed(kda_dtype dt, int B, int T, int H, int dk, int dv,
                                      const void *q, const void *k, const void *v,
                                      const void *g_raw, const void *beta,
                                      const float *init_state,
                                      const int32_t *cu_seqlens, int N,
                                      void *out, float *final_state,
                                      int checkpoint_every, float *checkpoints,
                                      long long checkpoint_rows,
                                      const kda_params *p, kda_stream_t stream);

/*
 * kda_chunk_fwd_split -- kda_chunk_fwd for launches with fewer (sequence,
 * head) chains than the GPU has multiprocessors.  Each sequence is cut into
 * consecutive segments of segment_tokens tokens (the last one shorter) that
 * run at the same time, and the exact result is assembled afterwards
 * ("Kimi K3: Two point eight trillion parameters, open weights, and
 * forty-seven pages of how", §The machine underneath: the sequence split
 * across the chip's multiprocessors and merged; the merge is the segment
 * composition of "Kimi K3：从三条信息流到完整系统", §FlashKDA 与 KCP, eq. (17)).
 * Because eq. (1) is affine in the state it starts from, a segment started
 * from S_in gives S_t = Phi_t S_in + S0_t and o_t = o0_t + S_in^T Phi_t^T q_t,
 * with (S0, o0) the segment run from a zero state and Phi_t the run with
 * v = 0 from the identity (its state is Phi_t, its output Phi_t^T q_t).  A
 * sequence of P segments therefore costs 2P - 1 concurrent chains of at most
 * segment_tokens tokens, plus a serial fp32 composition of P - 1 128 x 128
 * products per (sequence, head) and a per-token correction of the outputs
 * of segments 1 .. P - 1; it pays when N * H * (2P - 1) chains fit the GPU
 * at once (see kda_split_segment_tokens).
 *
 * Arguments as kda_chunk_fwd, plus:
 *   segment_tokens: a positive multiple of 16 (KDA_ERR_ARG otherwise).
 *   workspace: DEVICE scratch of at least kda_chunk_fwd_split_workspace(...)
 *          bytes, 256-byte aligned, caller-owned; its contents on entry are
 *          ignored and on return unspecified.  It must not overlap any other
 *          argument, and no other call may use it until this one completes
 *          on the stream.
 * Supported for dt = KDA_BF16 with dk = dv = 128 (the tensor-core prefill);
 * KDA_ERR_SHAPE otherwise.  Not combinable with checkpoints.
 * Numerics: the segments run the same kernel as kda_chunk_fwd; the
 * composition is fp32; for the tokens of segments 1 .. the zero-state and
 * transition runs write their outputs unrounded (fp32, in the workspace),
 * the correction S_in^T (Phi^T q) multiplies fp16 copies of S_in and of the
 * transition outputs with fp32 accumulation, and o is rounded to bf16 once.
 */
kda_status kda_chunk_fwd_split(kda_dtype dt, int B, int T, int H, int dk, int dv,
                               const void *q, const void *k, const void *v,
                               const void *g_raw, const void *beta,
                               const float *init_state,
                               const int32_t *cu_seqlens, int N, int segment_tokens,
                               void *out, float *final_state,
                               void *workspace, unsigned long long workspace_bytes,
                               const kda_params *p, kda_stream_t stream);

/*
 * kda_chunk_fwd_split_noalloc -- kda_chunk_fwd_split for callers that must
 * not allocate device memory: a process whose device memory is all handed
 * to its own caching pool, so that a cudaMalloc behind the pool's back can
 * fail or fragment it, or a plain C caller that has no device allocator of
 * its own.  The pages have no counterpart of this call: it is a packaging
 * of the segment split, not part of the method.
 *
 * Arguments, results and errors as kda_chunk_fwd_split without workspace:
 * the scratch is a buffer inside the library, KDA_SPLIT_SCRATCH_BYTES
 * (64 MiB) of device memory that every GPU which loads the library holds
 * until the process exits.  Sizes whose kda_chunk_fwd_split_workspace(...)
 * exceeds it return KDA_ERR_SCRATCH and enqueue nothing (for example 2
 * heads x 8192 tokens with 512-token segments need about 25 MiB; 96 heads x
 * 8192 tokens do not fit).  The caller still provides q, k, v, g_raw, beta,
 * init_state, out and final_state; nothing is allocated (no cudaMalloc,
 * cudaFree or allocating library call).
 *
 * The first call on a device looks up the buffer's device address (once
 * per device, with that device current); make that first call before any
 * stream capture.  Every call on a device shares the one buffer and leaves
 * its contents behind; each call writes every part of it that it reads, so
 * nothing has to start at zero.  Two calls whose work overlaps on the GPU
 * (different streams without ordering, or different host threads) race on
 * the buffer and produce wrong results: order them on one stream.
 */
#define KDA_SPLIT_SCRATCH_BYTES (64ull << 20)
kda_status kda_chunk_fwd_split_noalloc(kda_dtype dt, int B, int T, int H, int dk, int dv,
                                       const void *q, const void *k, const void *v,
                                       const void *g_raw, const void *beta,
                                       const float *init_state,
                                       const int32_t *cu_seqlens, int N, int segment_tokens,
                                       void *out, float *final_state,
                                       const kda_params *p, kda_stream_t stream);

/*
 * Sequence split across ranks (KCP: "Kimi K3：从三条信息流到完整系统",
 * §FlashKDA 与 KCP, eq. (17)): each of R ranks holds the next T tokens of the
 * same B sequences (rank 0 the first T).  Rank 0 runs kda_chunk_fwd from the
 * sequences' initial states; its final states are its pair.  Every rank
 * r >= 1 runs kda_chunk_fwd_kcp_part on its tokens, which yields its pair
 * (S0, Phi): the final state of its tokens run from a zero state, and the
 * transition Phi (its tokens run with v = 0 from the identity), so that the
 * state after its tokens is Phi S_in + S0 for the state S_in entering them.
 * The ranks exchange the pairs (an all-gather of B * 2 * H * dk * dk fp32
 * values per rank; the caller does it, e.g. with torch.distributed), then
 * every rank r >= 1 calls kda_chunk_fwd_kcp_finish with the pairs of ranks
 * 0 .. r: it composes S_in of its tokens by eq. (17) (fp32) and writes its
 * outputs o = o0 + S_in^T (Phi^T q) (rounded to bf16 once) and the state
 * after its tokens (the last rank's is the sequences' final state).
 * bf16 with dk = dv = 128 only (KDA_ERR_SHAPE otherwise); T >= 1.
 *
 * kda_chunk_fwd_kcp_workspace -- bytes of device workspace a rank needs
 *   (the same buffer, untouched in between, for its _part and _finish
 *   calls), or 0 for sizes the calls reject.  No GPU work.
 * kda_chunk_fwd_kcp_part -- q, k, g_raw [B, T, H, dk], v [B, T, H, dv],
 *   beta [B, T, H] (this rank's tokens, bf16); pair_out DEVICE fp32
 *   [B, 2, H, dk, dk], 16-byte aligned: [n][0] = S0, [n][1] = Phi.  Gate
 *   parameters as kda_chunk_fwd.  workspace 256-byte aligned.
 * kda_chunk_fwd_kcp_finish -- rank >= 1; pairs DEVICE fp32
 *   [rank + 1, B, 2, H, dk, dk] (entry [0][n][0] is rank 0's final state,
 *   [0][n][1] is not read); out [B, T, H, dv] bf16; final_state
 *   [B, H, dk, dv] fp32 or NULL.  Must follow the same rank's _part call on
 *   the same workspace (stream order).
 */
unsigned long long kda_chunk_fwd_kcp_workspace(int B, int T, int H, int dk, int dv);
kda_status kda_chunk_fwd_kcp_part(kda_dtype dt, int B, int T, int H, int dk, int dv,
                                  const void *q, const void *k, const void *v,
                                  const void *g_raw, const void *beta,
                                  float *pair_out, void *workspace, unsigned long long workspace_bytes,
                                  const kda_params *p, kda_stream_t stream);
kda_status kda_chunk_fwd_kcp_finish(int B, int T, int H, int dk, int dv, int rank,
                                    const float *pairs, void *out, float *final_state,
                                    void *workspace, unsigned long long workspace_bytes,
                                    kda_stream_t stream);

/*
 * kda_chunk_fwd_split_workspace -- bytes of workspace kda_chunk_fwd_split
 * needs for these sizes (B * T tokens in all, N sequences), or 0 for
 * arguments it would reject.  No GPU work.
 */
unsigned long long kda_chunk_fwd_split_workspace(int B, int T, int H, int dk, int dv, int N,
                                                 int segment_tokens);

/*
 * kda_split_segment_tokens -- host helper: a segment length (multiple of
 * 16) that puts every chain of the split in one wave on sm_count
 * multiprocessors (one chain per multiprocessor), or 0 when splitting
 * cannot (fewer than two segments per sequence fit).  varlen != 0: the
 * B * T tokens are N packed sequences of unknown lengths (the bound then
 * allows two chains more per sequence).  No GPU work.
 */
int kda_split_segment_tokens(int B, int T, int H, int N, int varlen, int sm_count);

/*
 * kda_checkpoint_rows -- host helper: rows of the checkpoint buffer for
 * these sequences (cu_seqlens_host: HOST [N+1] or NULL for B rows of T).
 * Returns -1 for arguments kda_chunk_fwd would reject (E not a positive
 * multiple of 16, a decreasing or out-of-range cu_seqlens).  No GPU work.
 */
long long kda_checkpoint_rows(int B, int T, const int32_t *cu_seqlens_host, int N,
                              int checkpoint_every);

/*
 * kda_decode_step -- advance N independent sequences by one token each.
 *
 * Inputs (dtype dt): q, k, g_raw [N, H, dk]; v [N, H, dv]; beta [N, H].
 * In/out: state [N, H, dk, dv] fp32, read and overwritten in place with the
 *         state after this token.
 * Output: out [N, H, dv] (dtype dt), o = scale * S_new^T q.
 * Each (sequence, head) state is read once and written once.
 */
kda_status kda_decode_step(kda_dtype dt, int N, int H, int dk, int dv,
                           const void *q, const void *k, const void *v,
                           const void *g_raw, const void *beta,
                           float *state, void *out,
                           const kda_params *p, kda_stream_t stream);

/* Name of the kernel kda_chunk_fwd launches for this dtype and head size
 * ("prefill_tc_kernel": tcgen05 tensor cores, bf16 with dk = dv = 128;
 * "prefill_simt_kernel": fp32 CUDA cores, every other supported case), or
 * NULL for an unsupported combination. */
const char *kda_chunk_fwd_kernel(kda_dtype dt, int dk, int dv);

/*
 * kda_decode_steps -- speculative replay: advance N sequences by up to K
 * drafted tokens each in one pass over the state.  Sequence n applies, in
 * order, its first accepted[n] tokens (clamped to [0, K]); the remaining
 * drafts leave no trace.  Only the drafts' projected inputs are kept, and
 * the accepted prefix is replayed on chip with no per-draft state copy
 * ("Kimi K3: Two point eight trillion parameters, open weights, and
 * forty-seven pages of how", §The machine underneath; "Kimi K3：从三条信息流到
 * 完整系统", §recurrent speculative decoding 不能复制整个状态).
 *
 * Inputs (dtype dt): q, k, g_raw [N, K, H, dk]; v [N, K, H, dv];
 *   beta [N, K, H]; accepted: DEVICE [N] int32, or NULL for all K.
 * In/out: state [N, H, dk, dv] fp32, read once and written once (left
 *   untouched for a sequence with accepted[n] == 0).
 * Output: out [N, K, H, dv]: o for every applied token; the rows of
 *   tokens that are not applied are not written.
 * kda_decode_step is the K = 1 case with every token applied.
 */
kda_status kda_decode_steps(kda_dtype dt, int N, int K, int H, int dk, int dv,
                            const void *q, const void *k, const void *v,
                            const void *g_raw, const void *beta, const int32_t *accepted,
                            float *state, void *out,
                            const kda_params *p, kda_stream_t stream);

/*
 * kda_qkv_prep -- the projection chain's tail before the operator
 * ("Kimi K3：从三条信息流到完整系统", §从投影到 Chunkwise 的完整接口, eq. (2)):
 *     q, k = L2Norm(Swish(ShortConv(x_q | x_k))),  v = Swish(ShortConv(x_v)),
 *     beta = Sigmoid(beta_logit)
 * ShortConv is the causal depthwise convolution of kernel size 4 along each
 * sequence's tokens, y_t = sum_i w[i] x_{t-3+i} per channel, no bias;
 * L2Norm divides each head's d channels by sqrt(sum x^2 + l2_eps).
 *
 * Inputs (dtype dt unless stated):
 *   x_qkv  [B, T, 3, H, d]  the q | k | v projections of each token.
 *   conv_w [3, H, d, 4] fp32: taps per channel, tap 3 multiplies x_t.
 *   beta_logit [B, T, H] or NULL (then beta must be NULL too).
 *   cu_seqlens / N: as kda_chunk_fwd (sequences are convolved separately).
 *   conv_state_in [N, 3, 3, H, d] or NULL (zeros): per sequence, the x_qkv
 *          rows of the three tokens before its first token, oldest first.
 * Outputs:
 *   q, k, v [B, T, H, d]; beta [B, T, H] (dtype dt).
 *   conv_state_out [N, 3, 3, H, d] or NULL: the last three x_qkv rows of
 *          each sequence (with conv_state_in rows where it is shorter than
 *          three), to continue it in a later call (decode: one token per
 *          sequence).  Must not alias conv_state_in.
 * l2_eps <= 0 selects 1e-6.
 */
kda_status kda_qkv_prep(kda_dtype dt, int B, int T, int H, int d,
                        const void *x_qkv, const float *conv_w, const void *beta_logit,
                        const int32_t *cu_seqlens, int N,
                        const void *conv_state_in, void *conv_state_out,
                        void *q, void *k, void *v, void *beta,
                        float l2_eps, kda_stream_t stream);

/*
 * kda_output_gate -- the output epilogue before W_o ("Kimi K3：从三条信息流到
 * 完整系统", §下界 log-decay 是一个 kernel 设计, eq. (6)):
 *     y = Sigmoid(gate) * RMSNorm(o),  RMSNorm(o) = o / sqrt(mean(o^2) + eps) * norm_w
 * over each row of d channels (one row = one token of one head).
 *   o, gate, y [rows, d] (dtype dt); norm_w [d] fp32 or NULL (ones).
 *   eps <= 0 selects 1e-5 (the model's rms_norm_eps).
 */
kda_status kda_output_gate(kda_dtype dt, long long rows, int d, const void *o, const void *gate,
                           const float *norm_w, float eps, void *y, kda_stream_t stream);

/* Static string for a status code (never NULL). */
const char *kda_status_str(kda_status s);

/* The CUDA error code (cudaError_t value) behind the last KDA_ERR_LAUNCH
 * returned on the calling host thread, or 0. */
int kda_last_cuda_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int kda_version(void);

/* Synchronises the current device, then reports whether any kernel of this
 * library gave up a bounded wait since the previous call (KDA_ERR_TIMEOUT;
 * the outputs of that launch are then unspecified) or the device reported an
 * error (KDA_ERR_LAUNCH).  Clears the timeout record.  The tensor-core
 * prefill bounds each of its internal waits at a few seconds and exits
 * instead of hanging. */
kda_status kda_check_device_status(void);

/* Exercises the failure report above without a real fault.  Enqueues one
 * small kernel on `stream` whose single thread waits, with the same bounded
 * wait the prefill and prep kernels use, on a shared-memory barrier that
 * nothing ever arrives at.  After `limit_us` microseconds the wait gives up
 * and records a timeout exactly as a stalled real launch would, so the next
 * kda_check_device_status() returns KDA_ERR_TIMEOUT and the one after it
 * KDA_OK.  The kernel starts no copy, tensor-core product or other
 * asynchronous work, so giving up leaves nothing in flight and the context
 * stays usable.  limit_us must be in [1, 100000] (KDA_ERR_ARG otherwise).
 * The pages define no such call: it is the library's own test hook for its
 * failure detection. */
kda_status kda_selftest_bounded_wait(int limit_us, kda_stream_t stream);

/* Number of CUDA kernels this library has enqueued in this process so far
 * (all entry points, all threads).  Lets a caller count launches over a
 * region of its own code. */
unsigned long long kda_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
