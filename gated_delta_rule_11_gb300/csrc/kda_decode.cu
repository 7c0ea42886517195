// Single-token KDA step ("a third kernel": decode), one CTA per (sequence,
// head).  The fp32 state S [dk, dv] (row = key channel c, column = value
// channel j) is streamed from HBM once and written back once, in place.
//
// Recurrence: "Kimi K3：从三条信息流到完整系统", §KDA 是带逐通道遗忘的 delta
// rule, eq. (1) in its expanded form.  With D = Diag(alpha) S:
//     a_j = sum_c alpha_c k_c S_cj      (= (D^T k)_j)
//     b_j = sum_c alpha_c q_c S_cj      (= (D^T q)_j)
//     u_j = beta (v_j - a_j)
//     S'_cj = alpha_c S_cj + k_c u_j
//     o_j = scale * (S'^T q)_j = scale * (b_j + (k.q) u_j)
// so both reductions happen in the single read pass, and the write pass
// needs only u.  alpha follows eq. (5) of §下界 log-decay 是一个 kernel 设计.
//
// Layout of the work: 256 threads; a row of S is dv/4 float4s; thread t
// owns float4 column (t % (dv/4)) of rows (t / (dv/4)) + m * rows_per_pass,
// holding its whole slice in registers between the two passes.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;

__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4 *p, float4 v) { __stcs(p, v); }

template <typename Tin, int DK, int DV>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_kernel(DecodeArgs a) {
    constexpr int V4 = DV / 4;                       // float4 per state row
    constexpr int RPP = kDecodeThreads / V4;         // rows per pass
    constexpr int PASSES = DK / RPP;
    static_assert(PASSES >= 1 && DK % RPP == 0, "tiling");

    __shared__ float s_alpha[DK], s_k[DK], s_ak[DK], s_aq[DK];
    __shared__ float s_v[DV];
    __shared__ __align__(16) float s_u[DV];
    __shared__ __align__(16) float s_red[2][RPP][DV];
    __shared__ float s_kq_part[DK / 32];

    const int tid = threadIdx.x;
    const int nh = blockIdx.x;                       // n * H + h
    const int h = nh % a.H;
    const int col4 = tid % V4;
    const int row0 = tid / V4;

    float4 *S = reinterpret_cast<float4 *>(a.state) + static_cast<size_t>(nh) * (DK * V4);

    // Issue the state loads first: they dominate the kernel's time.
    float4 st[PASSES];
#pragma unroll
    for (int m = 0; m < PASSES; ++m) st[m] = ld_stream(S + (row0 + m * RPP) * V4 + col4);

    const Tin *q = static_cast<const Tin *>(a.q) + static_cast<size_t>(nh) * DK;
    const Tin *k = static_cast<const Tin *>(a.k) + static_cast<size_t>(nh) * DK;
    const Tin *z = static_cast<const Tin *>(a.g) + static_cast<size_t>(nh) * DK;
    const Tin *v = static_cast<const Tin *>(a.v) + static_cast<size_t>(nh) * DV;
    const float beta = ld_in(static_cast<const Tin *>(a.beta) + nh);
    const float escale = a.A_log ? expf(__ldg(a.A_log + h)) : 1.0f;

    if (tid < DK) {
        const float kc = ld_in(k + tid), qc = ld_in(q + tid);
        const float alpha = expf(log_decay(ld_in(z + tid), escale, a.g_min));
        s_alpha[tid] = alpha;
        s_k[tid] = kc;
        s_ak[tid] = alpha * kc;
        s_aq[tid] = alpha * qc;
        float kq = kc * qc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
        if ((tid & 31) == 0) s_kq_part[tid >> 5] = kq;
    }
    if (tid < DV) s_v[tid] = ld_in(v + tid);
    __syncthreads();

    // Pass 1 (in registers): partial a_j and b_j over this thread's rows.
    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f), pb = pa;
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int c = row0 + m * RPP;
        const float ak = s_ak[c], aq = s_aq[c];
        pa.x += ak * st[m].x; pa.y += ak * st[m].y; pa.z += ak * st[m].z; pa.w += ak * st[m].w;
        pb.x += aq * st[m].x; pb.y += aq * st[m].y; pb.z += aq * st[m].z; pb.w += aq * st[m].w;
    }
    *reinterpret_cast<float4 *>(&s_red[0][row0][col4 * 4]) = pa;
    *reinterpret_cast<float4 *>(&s_red[1][row0][col4 * 4]) = pb;
    __syncthreads();

    if (tid < DV) {
        float av = 0.f, bv = 0.f;
#pragma unroll
        for (int r = 0; r < RPP; ++r) {
            av += s_red[0][r][tid];
            bv += s_red[1][r][tid];
        }
        float kq = 0.f;
#pragma unroll
        for (int w = 0; w < DK / 32; ++w) kq += s_kq_part[w];
        const float u = beta * (s_v[tid] - av);
        s_u[tid] = u;
        Tin *o = static_cast<Tin *>(a.out) + static_cast<size_t>(nh) * DV;
        st_out(o + tid, a.scale * (bv + kq * u));
    }
    __syncthreads();

    // Pass 2: S' = Diag(alpha) S + k u^T, written in place.
    const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[col4 * 4]);
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int c = row0 + m * RPP;
        const float al = s_alpha[c], kc = s_k[c];
        float4 r;
        r.x = al * st[m].x + kc * u4.x;
        r.y = al * st[m].y + kc * u4.y;
        r.z = al * st[m].z + kc * u4.z;
        r.w = al * st[m].w + kc * u4.w;
        st_stream(S + c * V4 + col4, r);
    }
}

template <typename Tin>
cudaError_t launch_t(int dk, int dv, const DecodeArgs &a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.N) * static_cast<unsigned>(a.H));
    const dim3 block(kDecodeThreads);
#define KDA_DEC_CASE(DK_, DV_)                                            \
    if (dk == DK_ && dv == DV_) {                                         \
        decode_kernel<Tin, DK_, DV_><<<grid, block, 0, s>>>(a);           \
        const cudaError_t e = cudaGetLastError();                         \
        if (e == cudaSuccess) count_launches(1);                          \
        return e;                                                         \
    }
    KDA_DEC_CASE(32, 32) KDA_DEC_CASE(32, 64) KDA_DEC_CASE(32, 128)
    KDA_DEC_CASE(64, 32) KDA_DEC_CASE(64, 64) KDA_DEC_CASE(64, 128)
    KDA_DEC_CASE(128, 32) KDA_DEC_CASE(128, 64) KDA_DEC_CASE(128, 128)
#undef KDA_DEC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(kda_dtype dt, int dk, int dv, const DecodeArgs &a, cudaStream_t s) {
    if (dt == KDA_BF16) return launch_t<__nv_bfloat16>(dk, dv, a, s);
    return launch_t<float>(dk, dv, a, s);
}

}  // namespace kda
