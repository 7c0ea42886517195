// Host side of the C ABI declared in include/kda.h: argument validation,
// kernel selection and launch on the caller's stream.  Nothing here
// allocates memory or synchronises.
#include <atomic>
#include <cstddef>
#include <cstdint>

#include "kda_internal.cuh"

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<unsigned long long> g_launches{0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool head_dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

void resolve_params(const kda_params *p, float &g_min, const float *&A_log, float &scale,
                    int &gate_mode, int &gate_scalar) {
    g_min = -5.0f;
    A_log = nullptr;
    scale = 1.0f;
    gate_mode = KDA_GATE_BOUNDED;
    gate_scalar = 0;
    if (p) {
        if (p->g_min != 0.0f) g_min = p->g_min;
        A_log = p->A_log;
        if (p->scale != 0.0f) scale = p->scale;
        gate_mode = p->gate_mode;
        gate_scalar = p->gate_per_head != 0;
    }
}

bool gate_mode_ok(const kda_params *p) {
    return !p || (p->gate_mode >= KDA_GATE_BOUNDED && p->gate_mode <= KDA_GATE_NONE);
}

// g_raw: required unless the gate is off; 16-byte aligned per channel,
// element-aligned per head.
kda_status check_gate(const kda_params *p, kda_dtype dt, const void *g_raw, bool needed) {
    if (!gate_mode_ok(p)) return KDA_ERR_ARG;
    const bool none = p && p->gate_mode == KDA_GATE_NONE;
    const bool scalar = p && p->gate_per_head;
    if (none) return KDA_OK;
    if (needed && !g_raw) return KDA_ERR_ARG;
    if (!g_raw) return KDA_OK;
    if (scalar) return aligned_to(g_raw, dt == KDA_F32 ? 4 : 2) ? KDA_OK : KDA_ERR_ALIGN;
    return aligned16(g_raw) ? KDA_OK : KDA_ERR_ALIGN;
}

kda_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    g_last_cuda_error = static_cast<int>(e);
    return KDA_ERR_LAUNCH;
}

}  // namespace

namespace kda {
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace kda

extern "C" {

const char *kda_status_str(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_ARG: return "invalid argument (null pointer, negative size or inconsistent N/B)";
        case KDA_ERR_DTYPE: return "unsupported dtype";
        case KDA_ERR_SHAPE: return "unsupported head dimension (dk and dv must be 32, 64 or 128)";
        case KDA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case KDA_ERR_LAUNCH: return "CUDA launch failed";
        case KDA_ERR_TIMEOUT: return "a bounded device wait timed out";
    }
    return "unknown status";
}

int kda_last_cuda_error(void) { return g_last_cuda_error; }

const char *kda_chunk_fwd_kernel(kda_dtype dt, int dk, int dv) {
    if ((dt != KDA_F32 && dt != KDA_BF16) || !head_dim_ok(dk) || !head_dim_ok(dv)) return nullptr;
    return kda::prefill_tc_supported(dt, dk, dv) ? "prefill_tc_kernel" : "prefill_simt_kernel";
}

int kda_version(void) { return 1 * 10000 + 0 * 100 + 0; }

unsigned long long kda_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

kda_status kda_check_device_status(void) {
    const cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        g_last_cuda_error = static_cast<int>(e);
        return KDA_ERR_LAUNCH;
    }
    const unsigned int waits = kda::take_tc_timeouts() + kda::take_prep_timeouts();
    return waits ? KDA_ERR_TIMEOUT : KDA_OK;
}

kda_status kda_selftest_bounded_wait(int limit_us, kda_stream_t stream) {
    if (limit_us < 1 || limit_us > 100000) return KDA_ERR_ARG;
    return from_cuda(kda::launch_wait_selftest(static_cast<uint64_t>(limit_us) * 1000u,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

long long kda_checkpoint_rows(int B, int T, const int32_t *cu_seqlens_host, int N,
                              int checkpoint_every) {
    if (checkpoint_every <= 0 || checkpoint_every % 16 != 0 || B < 0 || T < 0 || N < 0) return -1;
    if (!cu_seqlens_host) {
        if (N != B) return -1;
        return static_cast<long long>(B) * (T / checkpoint_every);
    }
    if (B != 1 || N < 1) return -1;
    long long rows = 0;
    for (int n = 0; n < N; ++n) {
        const long long len = static_cast<long long>(cu_seqlens_host[n + 1]) - cu_seqlens_host[n];
        if (len < 0 || cu_seqlens_host[n] < 0 || cu_seqlens_host[n + 1] > T) return -1;
        rows += len / checkpoint_every;
    }
    return rows;
}

kda_status kda_chunk_fwd_checkpointed(kda_dtype dt, int B, int T, int H, int dk, int dv,
                                      const void *q, const void *k, const void *v,
                                      const void *g_raw, const void *beta,
                                      const float *init_state,
                                      const int32_t *cu_seqlens, int N,
                                      void *out, float *final_state,
                                      int checkpoint_every, float *checkpoints,
                                      long long checkpoint_rows,
                                      const kda_params *p, kda_stream_t stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_DTYPE;
    if (B < 0 || T < 0 || H <= 0 || N < 0) return KDA_ERR_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDA_ERR_SHAPE;
    if (cu_seqlens) {
        if (B != 1 || N < 1) return KDA_ERR_ARG;
    } else if (N != B) {
        return KDA_ERR_ARG;
    }
    if (checkpoints && (checkpoint_every <= 0 || checkpoint_every % 16 != 0 || checkpoint_rows < 0))
        return KDA_ERR_ARG;
    const long long total = static_cast<long long>(B) * T;
    if (total > INT32_MAX || static_cast<long long>(N) * H > INT32_MAX) return KDA_ERR_ARG;
    if (total > 0 && (!q || !k || !v || !beta || !out)) return KDA_ERR_ARG;
    const void *ptrs[] = {q, k, v, init_state, out, final_state, checkpoints};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGN;
    if (!aligned_to(beta, dt == KDA_F32 ? 4 : 2) || !aligned_to(cu_seqlens, 4)) return KDA_ERR_ALIGN;
    if (const kda_status gs = check_gate(p, dt, g_raw, total > 0)) return gs;
    if (N == 0 || (total == 0 && !final_state)) return KDA_OK;  // nothing to compute

    kda::PrefillArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g_raw; a.beta = beta;
    a.init_state = init_state;
    a.cu_seqlens = cu_seqlens;
    a.out = out;
    a.final_state = final_state;
    const bool ck = checkpoints && checkpoint_rows > 0;
    a.ckpt = ck ? checkpoints : nullptr;
    a.ckpt_rows = ck ? checkpoint_rows : 0;
    a.ckpt_every = ck ? checkpoint_every : 0;
    resolve_params(p, a.g_min, a.A_log, a.scale, a.gate_mode, a.gate_scalar);
    if (a.A_log && !aligned_to(a.A_log, 4)) return KDA_ERR_ALIGN;
    a.N = N;
    a.H = H;
    a.T_total = static_cast<int>(total);
    a.T_seq = T;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // every gate map runs on the tensor cores (an unbounded map's tiles past
    // fp32's range take the kernel's position-pair path for L and A)
    if (kda::prefill_tc_supported(dt, dk, dv) && a.T_total > 0)
        return from_cuda(kda::launch_prefill_tc(a, s));
    return from_cuda(kda::launch_prefill_simt(dt, dk, dv, a, s));
}

kda_status kda_chunk_fwd(kda_dtype dt, int B, int T, int H, int dk, int dv,
                         const void *q, const void *k, const void *v,
                         const void *g_raw, const void *beta,
                         const float *init_state,
                         const int32_t *cu_seqlens, int N,
                         void *out, float *final_state,
                         const kda_params *p, kda_stream_t stream) {
    return kda_chunk_fwd_checkpointed(dt, B, T, H, dk, dv, q, k, v, g_raw, beta, init_state,
                                      cu_seqlens, N, out, final_state, 0, nullptr, 0, p, stream);
}

kda_status kda_decode_steps(kda_dtype dt, int N, int K, int H, int dk, int dv,
                            const void *q, const void *k, const void *v,
                            const void *g_raw, const void *beta, const int32_t *accepted,
                            float *state, void *out,
                            const kda_params *p, kda_stream_t stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_DTYPE;
    if (N < 0 || K < 1 || H <= 0) return KDA_ERR_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDA_ERR_SHAPE;
    if (static_cast<long long>(N) * H > INT32_MAX || static_cast<long long>(N) * K * H > INT32_MAX)
        return KDA_ERR_ARG;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !beta || !state || !out) return KDA_ERR_ARG;
    const void *ptrs[] = {q, k, v, state, out};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr)) return KDA_ERR_ALIGN;
    if (!aligned_to(beta, dt == KDA_F32 ? 4 : 2) || !aligned_to(accepted, 4)) return KDA_ERR_ALIGN;
    if (const kda_status gs = check_gate(p, dt, g_raw, true)) return gs;
    kda::DecodeArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g_raw; a.beta = beta;
    a.accepted = accepted;
    a.state = state;
    a.out = out;
    resolve_params(p, a.g_min, a.A_log, a.scale, a.gate_mode, a.gate_scalar);
    if (a.A_log && !aligned_to(a.A_log, 4)) return KDA_ERR_ALIGN;
    a.N = N;
    a.K = K;
    a.H = H;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return from_cuda(kda::launch_decode(dt, dk, dv, a, s));
}

kda_status kda_decode_step(kda_dtype dt, int N, int H, int dk, int dv,
                           const void *q, const void *k, const void *v,
                           const void *g_raw, const void *beta,
                           float *state, void *out,
                           const kda_params *p, kda_stream_t stream) {
    return kda_decode_steps(dt, N, 1, H, dk, dv, q, k, v, g_raw, beta, nullptr, state, out, p, stream);
}

kda_status kda_qkv_prep(kda_dtype dt, int B, int T, int H, int d,
                        const void *x_qkv, const float *conv_w, const void *beta_logit,
                        const int32_t *cu_seqlens, int N,
                        const void *conv_state_in, void *conv_state_out,
                        void *q, void *k, void *v, void *beta,
                        float l2_eps, kda_stream_t stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_DTYPE;
    if (B < 0 || T < 0 || H <= 0 || N < 0) return KDA_ERR_ARG;
    if (!head_dim_ok(d)) return KDA_ERR_SHAPE;
    if (cu_seqlens) {
        if (B != 1 || N < 1) return KDA_ERR_ARG;
    } else if (N != B) {
        return KDA_ERR_ARG;
    }
    const long long total = static_cast<long long>(B) * T;
    if (total > INT32_MAX || static_cast<long long>(N) * 3 * H * d > INT32_MAX) return KDA_ERR_ARG;
    if (total > 0 && (!x_qkv || !conv_w || !q || !k || !v)) return KDA_ERR_ARG;
    if ((beta_logit == nullptr) != (beta == nullptr)) return KDA_ERR_ARG;
    const void *ptrs[] = {x_qkv, conv_w, conv_state_in, conv_state_out, q, k, v};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGN;
    const uintptr_t es = dt == KDA_F32 ? 4 : 2;
    if (!aligned_to(beta_logit, es) || !aligned_to(beta, es) || !aligned_to(cu_seqlens, 4))
        return KDA_ERR_ALIGN;
    if (N == 0 || (total == 0 && !conv_state_out)) return KDA_OK;
    kda::PrepArgs a;
    a.x = x_qkv; a.conv_w = conv_w; a.beta_logit = beta_logit;
    a.cu_seqlens = cu_seqlens;
    a.state_in = conv_state_in; a.state_out = conv_state_out;
    a.q = q; a.k = k; a.v = v; a.beta = beta;
    a.N = N; a.H = H; a.T_total = static_cast<int>(total); a.T_seq = T;
    a.l2_eps = l2_eps > 0.f ? l2_eps : 1e-6f;
    return from_cuda(kda::launch_prep(dt, d, a, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_output_gate(kda_dtype dt, long long rows, int d, const void *o, const void *gate,
                           const float *norm_w, float eps, void *y, kda_stream_t stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_DTYPE;
    if (rows < 0) return KDA_ERR_ARG;
    if (!head_dim_ok(d)) return KDA_ERR_SHAPE;
    if (rows == 0) return KDA_OK;
    if (!o || !gate || !y) return KDA_ERR_ARG;
    const void *ptrs[] = {o, gate, y};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr)) return KDA_ERR_ALIGN;
    if (!aligned_to(norm_w, 4)) return KDA_ERR_ALIGN;
    kda::PostArgs a;
    a.o = o; a.gate = gate; a.norm_w = norm_w; a.y = y;
    a.rows = rows;
    a.eps = eps > 0.f ? eps : 1e-5f;
    return from_cuda(kda::launch_output_gate(dt, d, a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
