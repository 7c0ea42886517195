// Internal declarations shared by the libkda translation units.
// Not part of the public ABI (that is include/kda.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Per-launch arguments of the prefill kernels.  Token-major packed layout:
// q, k, g_raw [T_total, H, dk]; v, out [T_total, H, dv]; beta [T_total, H];
// states [N, H, dk, dv] fp32.
struct PrefillArgs {
    const void *q, *k, *v, *g, *beta;
    const float *init_state;
    const int32_t *cu_seqlens;  // device [N+1] or nullptr (then fixed length T_seq)
    void *out;
    float *final_state;
    const float *A_log;         // device [H] or nullptr
    int N, H, T_total, T_seq;
    float g_min, scale;
    int gate_mode, gate_scalar;  // kda_gate_mode; 1 = one gate per (token, head)
    // State checkpoints: every ckpt_every tokens of each sequence (a multiple
    // of 16; 0 = none) into ckpt [ckpt_rows, H, dk, dv]; rows at or past
    // ckpt_rows are never written.
    float *ckpt;
    long long ckpt_rows;
    int ckpt_every;
    // Segment split (tensor-core prefill only; ckpt unused): when vseg is
    // set, chain c runs the virtual sequence vseg[c / H] = {first token,
    // end token, VSEG_* flags, init source} instead of sequence c / H, and
    // final_state has one slot per virtual chain.  Every virtual chain
    // writes its output rows unrounded, as fp32: to out_trans when flagged
    // VSEG_OUT_TRANS, else to out_zero ([T_total, H, 128] each); out is not
    // written.
    const int4 *vseg;
    float *out_trans, *out_zero;
};

// Flags of a virtual sequence (PrefillArgs::vseg[].z).
enum : int {
    VSEG_ZERO_INIT = 1,   // the state entering it is zero (init_state ignored)
    VSEG_IDENT_INIT = 2,  // the state entering it is the identity (dk == dv)
    VSEG_ZERO_V = 4,      // every value is zero (V loaded past the last head: TMA zero fill)
    VSEG_OUT_TRANS = 8,   // its output rows go to out_trans (fp32)
    VSEG_OUT_ZERO = 16,   // its output rows go to out_zero (fp32)
    VSEG_EMPTY = 32,      // no chain: the CTA exits at once
    VSEG_OUT_FINAL = 64   // its out_zero rows are the outputs themselves (a sequence's first
                          // segment): the fixup only rounds them
};

// Decode: q, k, g_raw [N, K, H, dk]; v, out [N, K, H, dv]; beta [N, K, H];
// sequence n applies its first accepted[n] tokens (all K when accepted is null).
struct DecodeArgs {
    const void *q, *k, *v, *g, *beta;
    const int32_t *accepted;
    float *state;
    void *out;
    const float *A_log;
    int N, K, H;
    float g_min, scale;
    int gate_mode, gate_scalar;
};

// Element loads/stores in the caller's dtype, computed in fp32.
template <typename T> __device__ __forceinline__ float ld_in(const T *p);
template <> __device__ __forceinline__ float ld_in<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(__ldg(p));
}
template <typename T> __device__ __forceinline__ void st_out(T *p, float x);
template <> __device__ __forceinline__ void st_out<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
}

// Bounded log-decay, "Kimi K3：从三条信息流到完整系统" §下界 log-decay 是一个
// kernel 设计, eq. (5): g = g_min * sigmoid(e^A z); escale = e^A.
__device__ __forceinline__ float log_decay(float z, float escale, float g_min) {
    return g_min / (1.0f + expf(-escale * z));
}

// Pre/post passes.  prep: x [T, 3, H, d] (q | k | v projections), conv_w
// [3, H, d, 4] fp32, beta_logit [T, H], conv states [N, 3, 3, H, d] (the
// last three tokens' x, oldest first); outputs q, k, v [T, H, d], beta
// [T, H].  post: o, gate, y [rows, d], norm_w [d] fp32.
struct PrepArgs {
    const void *x;
    const float *conv_w;
    const void *beta_logit;
    const int32_t *cu_seqlens;
    const void *state_in;
    void *state_out;
    void *q, *k, *v, *beta;
    int N, H, T_total, T_seq;
    float l2_eps;
};
struct PostArgs {
    const void *o, *gate;
    const float *norm_w;
    void *y;
    long long rows;
    float eps;
};
cudaError_t launch_prep(kda_dtype dt, int d, const PrepArgs &a, cudaStream_t s);
cudaError_t launch_output_gate(kda_dtype dt, int d, const PostArgs &a, cudaStream_t s);

// Log-decay g of one gate input under each kda_gate_mode.  The negative
// softplus is -(max(x, 0) + log(1 + e^-|x|)), which never overflows.
__device__ __forceinline__ float gate_log_decay(int mode, float z, float escale, float g_min) {
    switch (mode) {
    case KDA_GATE_BOUNDED: return log_decay(z, escale, g_min);
    case KDA_GATE_LOG_DECAY: return z;
    case KDA_GATE_NEG_SOFTPLUS: {
        const float x = escale * z;
        return -(fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
    }
    default: return 0.f;
    }
}

// Sequence span [bos, eos) of sequence n, clamped into [0, T_total].
__device__ __forceinline__ void seq_span(const PrefillArgs &a, int n, int &bos, int &eos) {
    if (a.cu_seqlens) {
        int b0 = a.cu_seqlens[n], e0 = a.cu_seqlens[n + 1];
        b0 = min(max(b0, 0), a.T_total);
        e0 = min(max(e0, b0), a.T_total);
        bos = b0;
        eos = e0;
    } else {
        bos = n * a.T_seq;
        eos = bos + a.T_seq;
    }
}

// Row of sequence n's first checkpoint: the checkpoints of sequences 0..n-1
// (floor(length / ckpt_every) each).  Called by whole warps.
__device__ __forceinline__ long long ckpt_first_row(const PrefillArgs &a, int n) {
    if (!a.cu_seqlens) return static_cast<long long>(n) * (a.T_seq / a.ckpt_every);
    long long cnt = 0;
    for (int m = threadIdx.x & 31; m < n; m += 32) {
        int b, e;
        seq_span(a, m, b, e);
        cnt += (e - b) / a.ckpt_every;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    return cnt;
}

// Checkpoint slot after `done` tokens of a sequence whose first checkpoint
// row is `row0`, or nullptr when no checkpoint falls there or the row is past
// the buffer.
__device__ __forceinline__ float *ckpt_slot(const PrefillArgs &a, long long row0, int done, int h,
                                            size_t state_elems) {
    if (!a.ckpt || done <= 0 || done % a.ckpt_every != 0) return nullptr;
    const long long row = row0 + done / a.ckpt_every - 1;
    if (row >= a.ckpt_rows) return nullptr;
    return a.ckpt + (static_cast<size_t>(row) * a.H + h) * state_elems;
}

// Record n successfully enqueued kernels (backs kda_launch_count).
void count_launches(unsigned n);

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_decode(kda_dtype dt, int dk, int dv, const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_prefill_simt(kda_dtype dt, int dk, int dv, const PrefillArgs &a,
                                cudaStream_t s);

// Tensor-core prefill (bf16, dk = dv = 128).
bool prefill_tc_supported(kda_dtype dt, int dk, int dv);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s);
// Number of bounded device waits that gave up since the last call (syncs the device).
unsigned int take_tc_timeouts();
unsigned int take_prep_timeouts();
// Test hook: one kernel whose bounded wait on a never-arriving barrier gives up.
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s);

// Segment split (kda_split.cu).  Workspace carved by the caller:
//   vseg [nv_max] int4, seqtab [N] int2 {first virtual index, segments},
//   states [nv_max, H, d, d] fp32 (the virtual chains' final states),
//   s_in [nv_max, H, d, d] fp32 (the true state entering each segment),
//   out_trans, out_zero [T_total, H, d] fp32 (the transition runs' and the
//   zero-state runs' outputs of the tokens of segments 1..).
struct SplitArgs {
    int N, H, T_total, T_seq, seg_tokens, nv_max;
    const int32_t *cu_seqlens;
    int4 *vseg;
    int2 *seqtab;
    float *states, *s_in;
    float *out_trans, *out_zero;
    void *out;            // the call's output rows (segments 1.. written by the fixup)
    float *final_state;   // [N, H, d, d] or nullptr
};
cudaError_t launch_split_plan(const SplitArgs &a, cudaStream_t s);

// Sequence split across ranks (kda_chunk_fwd_kcp_part / _finish): B
// sequences of T tokens on this rank; workspace: vseg [2B] int4, s_in
// [B, H, d, d] fp32, out_trans, out_zero [B T, H, d] fp32.
struct KcpArgs {
    int B, T, H, rank;
    int4 *vseg;
    float *s_in, *out_trans, *out_zero;
    const float *pairs;   // [rank + 1, B, 2, H, d, d]
    void *out;            // [B T, H, d] bf16
    float *final_state;   // [B, H, d, d] or nullptr
};
cudaError_t launch_kcp_plan(const KcpArgs &a, cudaStream_t s);
cudaError_t launch_kcp_finish(const KcpArgs &a, cudaStream_t s);
cudaError_t launch_split_compose(const SplitArgs &a, cudaStream_t s);
cudaError_t launch_split_fixup(const SplitArgs &a, cudaStream_t s);

}  // namespace kda
