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
        case KDA_ERR_SCRATCH: return "the call needs more scratch than the library's static buffer (KDA_SPLIT_SCRATCH_BYTES) holds";
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

    kda::PrefillArgs a{};
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

// ---------------------------------------------------------------- segment split
namespace {
constexpr size_t kSplitAlign = 256;
size_t round_up(size_t x) { return (x + kSplitAlign - 1) / kSplitAlign * kSplitAlign; }

// Upper bound of the virtual sequences: sum over n of (2 P_n - 1) with
// P_n = max(1, ceil(L_n / tau)) <= L_n / tau + 1.
long long split_nv_max(long long total, int N, int tau) { return 2 * (total / tau) + 2 + N; }

struct SplitLayout {
    size_t vseg, seqtab, states, s_in, out_trans, out_zero, bytes;
};
SplitLayout split_layout(long long total, int H, int N, int tau) {
    const long long nv = split_nv_max(total, N, tau);
    const size_t state_bytes = static_cast<size_t>(nv) * H * 128 * 128 * sizeof(float);
    SplitLayout l;
    l.vseg = 0;
    l.seqtab = round_up(l.vseg + static_cast<size_t>(nv) * 16);
    l.states = round_up(l.seqtab + static_cast<size_t>(N) * 8);
    l.s_in = round_up(l.states + state_bytes);
    const size_t rows = static_cast<size_t>(total) * H * 128 * sizeof(float);
    l.out_trans = round_up(l.s_in + state_bytes);
    l.out_zero = round_up(l.out_trans + rows);
    l.bytes = round_up(l.out_zero + rows);
    return l;
}
}  // namespace

unsigned long long kda_chunk_fwd_split_workspace(int B, int T, int H, int dk, int dv, int N,
                                                 int segment_tokens) {
    if (B < 0 || T < 0 || H <= 0 || N < 1 || dk != 128 || dv != 128 || segment_tokens <= 0 ||
        segment_tokens % 16 != 0)
        return 0;
    return split_layout(static_cast<long long>(B) * T, H, N, segment_tokens).bytes;
}

int kda_split_segment_tokens(int B, int T, int H, int N, int varlen, int sm_count) {
    if (B < 0 || T < 0 || H <= 0 || N < 1 || sm_count < 1) return 0;
    const long long chains = static_cast<long long>(N) * H;
    // P segments per sequence put N H (2P - 1) chains in one wave; packed
    // sequences of unequal length may need up to N H (2P + 1).
    const long long per = sm_count / chains;
    const long long P = varlen ? (per - 1) / 2 : (per + 1) / 2;
    if (P < 2) return 0;
    const long long total = static_cast<long long>(B) * T;
    const long long len = varlen ? (total + N - 1) / N : T;   // mean sequence length
    const long long tau = ((len + P - 1) / P + 15) / 16 * 16;
    if (tau <= 0 || tau >= len) return 0;
    return static_cast<int>(tau);
}

kda_status kda_chunk_fwd_split(kda_dtype dt, int B, int T, int H, int dk, int dv,
                               const void *q, const void *k, const void *v,
                               const void *g_raw, const void *beta,
                               const float *init_state,
                               const int32_t *cu_seqlens, int N, int segment_tokens,
                               void *out, float *final_state,
                               void *workspace, unsigned long long workspace_bytes,
                               const kda_params *p, kda_stream_t stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_DTYPE;
    if (B < 0 || T < 0 || H <= 0 || H > 65535 || N < 0) return KDA_ERR_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return KDA_ERR_SHAPE;
    if (!kda::prefill_tc_supported(dt, dk, dv)) return KDA_ERR_SHAPE;   // bf16, dk = dv = 128 only
    if (segment_tokens <= 0 || segment_tokens % 16 != 0) return KDA_ERR_ARG;
    if (cu_seqlens) {
        if (B != 1 || N < 1) return KDA_ERR_ARG;
    } else if (N != B) {
        return KDA_ERR_ARG;
    }
    const long long total = static_cast<long long>(B) * T;
    if (total > INT32_MAX || N == 0) return kda_chunk_fwd(dt, B, T, H, dk, dv, q, k, v, g_raw, beta,
                                                          init_state, cu_seqlens, N, out, final_state,
                                                          p, stream);
    const long long nv = split_nv_max(total, N, segment_tokens);
    if (nv * H > INT32_MAX) return KDA_ERR_ARG;
    if (total == 0)   // nothing to split: the plain call copies the initial states
        return kda_chunk_fwd(dt, B, T, H, dk, dv, q, k, v, g_raw, beta, init_state, cu_seqlens, N,
                             out, final_state, p, stream);
    if (!q || !k || !v || !beta || !out || !workspace) return KDA_ERR_ARG;
    const void *ptrs[] = {q, k, v, init_state, out, final_state};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGN;
    if (!aligned_to(workspace, kSplitAlign)) return KDA_ERR_ALIGN;
    if (!aligned_to(beta, 2) || !aligned_to(cu_seqlens, 4)) return KDA_ERR_ALIGN;
    if (const kda_status gs = check_gate(p, dt, g_raw, true)) return gs;
    const SplitLayout l = split_layout(total, H, N, segment_tokens);
    if (workspace_bytes < l.bytes) return KDA_ERR_ARG;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    kda::SplitArgs sa;
    sa.N = N;
    sa.H = H;
    sa.T_total = static_cast<int>(total);
    sa.T_seq = T;
    sa.seg_tokens = segment_tokens;
    sa.nv_max = static_cast<int>(nv);
    sa.cu_seqlens = cu_seqlens;
    sa.vseg = reinterpret_cast<int4 *>(ws + l.vseg);
    sa.seqtab = reinterpret_cast<int2 *>(ws + l.seqtab);
    sa.states = reinterpret_cast<float *>(ws + l.states);
    sa.s_in = reinterpret_cast<float *>(ws + l.s_in);
    sa.out_trans = reinterpret_cast<float *>(ws + l.out_trans);
    sa.out_zero = reinterpret_cast<float *>(ws + l.out_zero);
    sa.out = out;
    sa.final_state = final_state;

    kda::PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g_raw; a.beta = beta;
    a.init_state = init_state;
    a.out = out;
    a.final_state = sa.states;
    resolve_params(p, a.g_min, a.A_log, a.scale, a.gate_mode, a.gate_scalar);
    if (a.A_log && !aligned_to(a.A_log, 4)) return KDA_ERR_ALIGN;
    a.N = sa.nv_max;
    a.H = H;
    a.T_total = sa.T_total;
    a.T_seq = T;
    a.vseg = sa.vseg;
    a.out_trans = sa.out_trans;
    a.out_zero = sa.out_zero;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (const kda_status st = from_cuda(kda::launch_split_plan(sa, s))) return st;
    if (const kda_status st = from_cuda(kda::launch_prefill_tc(a, s))) return st;
    if (const kda_status st = from_cuda(kda::launch_split_compose(sa, s))) return st;
    return from_cuda(kda::launch_split_fixup(sa, s));
}

// ---------------------------------------------------------------- sequence split across ranks
namespace {
struct KcpLayout {
    size_t vseg, s_in, out_trans, out_zero, bytes;
};
KcpLayout kcp_layout(int B, int T, int H) {
    const size_t rows = static_cast<size_t>(B) * T * H * 128 * sizeof(float);
    KcpLayout l;
    l.vseg = 0;
    l.s_in = round_up(static_cast<size_t>(2) * B * 16);
    l.out_trans = round_up(l.s_in + static_cast<size_t>(B) * H * 128 * 128 * sizeof(float));
    l.out_zero = round_up(l.out_trans + rows);
    l.bytes = round_up(l.out_zero + rows);
    return l;
}
bool kcp_sizes_ok(int B, int T, int H, int dk, int dv) {
    return B >= 1 && T >= 1 && H >= 1 && H <= 65535 && dk == 128 && dv == 128 &&
           static_cast<long long>(B) * T <= INT32_MAX && 2LL * B * H <= INT32_MAX;
}
kda::KcpArgs kcp_args(int B, int T, int H, void *workspace) {
    const KcpLayout l = kcp_layout(B, T, H);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    kda::KcpArgs k{};
    k.B = B;
    k.T = T;
    k.H = H;
    k.vseg = reinterpret_cast<int4 *>(ws + l.vseg);
    k.s_in = reinterpret_cast<float *>(ws + l.s_in);
    k.out_trans = reinterpret_cast<float *>(ws + l.out_trans);
    k.out_zero = reinterpret_cast<float *>(ws + l.out_zero);
    return k;
}
}  // namespace

unsigned long long kda_chunk_fwd_kcp_workspace(int B, int T, int H, int dk, int dv) {
    return kcp_sizes_ok(B, T, H, dk, dv) ? kcp_layout(B, T, H).bytes : 0;
}

kda_status kda_chunk_fwd_kcp_part(kda_dtype dt, int B, int T, int H, int dk, int dv,
                                  const void *q, const void *k, const void *v,
                                  const void *g_raw, const void *beta,
                                  float *pair_out, void *workspace, unsigned long long workspace_bytes,
                                  const kda_params *p, kda_stream_t stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_DTYPE;
    if (B < 0 || T < 0 || H <= 0) return KDA_ERR_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv) || !kda::prefill_tc_supported(dt, dk, dv)) return KDA_ERR_SHAPE;
    if (!kcp_sizes_ok(B, T, H, dk, dv)) return KDA_ERR_ARG;
    const long long total = static_cast<long long>(B) * T;
    if (!pair_out || !workspace || !q || !k || !v || !beta) return KDA_ERR_ARG;
    const void *ptrs[] = {q, k, v, pair_out};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGN;
    if (!aligned_to(workspace, kSplitAlign) || !aligned_to(beta, 2)) return KDA_ERR_ALIGN;
    if (const kda_status gs = check_gate(p, dt, g_raw, true)) return gs;
    if (workspace_bytes < kcp_layout(B, T, H).bytes) return KDA_ERR_ARG;
    kda::KcpArgs ka = kcp_args(B, T, H, workspace);
    kda::PrefillArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g_raw; a.beta = beta;
    // every virtual sequence writes fp32 rows (out_zero / out_trans), so the
    // bf16 output map is never stored through; it describes a valid region
    a.out = ka.out_zero;
    a.final_state = pair_out;    // slot 2n + w of [B, 2, H, d, d]: w = 0 zero-state run, 1 transition
    resolve_params(p, a.g_min, a.A_log, a.scale, a.gate_mode, a.gate_scalar);
    if (a.A_log && !aligned_to(a.A_log, 4)) return KDA_ERR_ALIGN;
    a.N = 2 * B;
    a.H = H;
    a.T_total = static_cast<int>(total);
    a.T_seq = T;
    a.vseg = ka.vseg;
    a.out_trans = ka.out_trans;
    a.out_zero = ka.out_zero;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (const kda_status st = from_cuda(kda::launch_kcp_plan(ka, s))) return st;
    return from_cuda(kda::launch_prefill_tc(a, s));
}

kda_status kda_chunk_fwd_kcp_finish(int B, int T, int H, int dk, int dv, int rank,
                                    const float *pairs, void *out, float *final_state,
                                    void *workspace, unsigned long long workspace_bytes,
                                    kda_stream_t stream) {
    if (!kcp_sizes_ok(B, T, H, dk, dv) || rank < 1) return dk == 128 && dv == 128 ? KDA_ERR_ARG : KDA_ERR_SHAPE;
    if (!pairs || !workspace || !out) return KDA_ERR_ARG;
    const void *ptrs[] = {pairs, out, final_state};
    for (const void *ptr : ptrs)
        if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGN;
    if (!aligned_to(workspace, kSplitAlign)) return KDA_ERR_ALIGN;
    if (workspace_bytes < kcp_layout(B, T, H).bytes) return KDA_ERR_ARG;
    kda::KcpArgs ka = kcp_args(B, T, H, workspace);
    ka.rank = rank;
    ka.pairs = pairs;
    ka.out = out;
    ka.final_state = final_state;
    return from_cuda(kda::launch_kcp_finish(ka, reinterpret_cast<cudaStream_t>(stream)));
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
