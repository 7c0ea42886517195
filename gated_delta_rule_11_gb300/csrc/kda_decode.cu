// KDA decode: each (sequence, head) advances by the first `accepted` of K
// drafted tokens in one pass over its state (K = 1, all accepted: the plain
// single-token step, "a third kernel" of "Kimi K3: Two point eight trillion
// parameters, open weights, and forty-seven pages of how", §The machine
// underneath).  Replaying only the accepted prefix of speculative drafts on
// chip, with no per-draft state copy, is the scheme of that section and of
// "Kimi K3：从三条信息流到完整系统", §recurrent speculative decoding 不能复制整个状态.
// The gate input becomes alpha under any kda_gate_mode (eq. (5) by
// default), one gate per key channel or one per head.
// One CTA per (sequence, head); the fp32 state S [dk, dv] (row = key channel
// c, column = value channel j) is read from HBM once, kept in registers
// across the tokens, and written back once, in place.
//
// Recurrence: "Kimi K3：从三条信息流到完整系统", §KDA 是带逐通道遗忘的 delta
// rule, eq. (1) in its expanded form.  Per token, with D = Diag(alpha) S:
//     a_j = sum_c alpha_c k_c S_cj      (= (D^T k)_j)
//     b_j = sum_c alpha_c q_c S_cj      (= (D^T q)_j)
//     u_j = beta (v_j - a_j)
//     S'_cj = alpha_c S_cj + k_c u_j
//     o_j = scale * (S'^T q)_j = scale * (b_j + (k.q) u_j)
// so both reductions happen in a single pass over the state.  alpha follows
// eq. (5) of §下界 log-decay 是一个 kernel 设计.
//
// Two kernels, both with the state in registers as float4 column groups of
// whole rows (256 threads): decode1_kernel, the single-token step over all
// dv columns, combining the two reductions over c across warps through
// shared memory; decode_kernel, the multi-token replay, over one dv/CS-column
// slab per CTA with one cross-warp reduction per token.  The replay's
// per-token channel vectors (alpha k, alpha q) and (alpha, k) (8-byte pairs,
// one load per row, widened to the packed two-lane form in registers), v, beta and
// k.q are computed for a block of up to 8 tokens at once into shared memory,
// with their loads in flight beside the state's (bf16 drafts are first
// staged into shared memory by cp.async).
#include "kda_internal.cuh"
#include "kda_sm100.cuh"
#include "kda_tc_util.cuh"

namespace kda {
namespace {
using sm100::f32x2;
using sm100::pack2;
using sm100::unpack2;
using sm100::ffma2;
using sm100::fmul2;

constexpr int kDecodeThreads = 256;
constexpr int kTokBlock = 8;                         // tokens prepared per barrier

__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
// 16-byte global -> shared copy that holds no registers while in flight
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void st_stream(float4 *p, float4 v) { __stcs(p, v); }

// Single-token step with whole rows per warp (a warp instruction touches one
// 512-byte row of S): rows row0 + m * RPP per thread, the reductions over c
// combined across warps through shared memory.  K = 1, every token applied.
// GenericGate = false compiles the default gate (eq. (5), per channel) with
// its input load issued beside the others; true takes any kda_gate_mode.
template <typename Tin, int DK, int DV, bool GenericGate>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode1_kernel(DecodeArgs a) {
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
    float4 st[PASSES];
#pragma unroll
    for (int m = 0; m < PASSES; ++m) st[m] = ld_stream(S + (row0 + m * RPP) * V4 + col4);

    const Tin *q = static_cast<const Tin *>(a.q) + static_cast<size_t>(nh) * DK;
    const Tin *k = static_cast<const Tin *>(a.k) + static_cast<size_t>(nh) * DK;
    // gate input of key channel c: per channel [N, H, dk] or per head [N, H]
    const Tin *z = static_cast<const Tin *>(a.g) + (a.gate_scalar ? static_cast<size_t>(nh)
                                                                   : static_cast<size_t>(nh) * DK);
    const Tin *v = static_cast<const Tin *>(a.v) + static_cast<size_t>(nh) * DV;
    const float beta = ld_in(static_cast<const Tin *>(a.beta) + nh);
    const float escale = a.A_log ? expf(__ldg(a.A_log + h)) : 1.0f;

    if (tid < DK) {
        const float kc = ld_in(k + tid), qc = ld_in(q + tid);
        float alpha;
        if constexpr (GenericGate) {
            const float zc = a.gate_mode == KDA_GATE_NONE ? 0.f : ld_in(z + (a.gate_scalar ? 0 : tid));
            alpha = expf(gate_log_decay(a.gate_mode, zc, escale, a.g_min));
        } else {
            alpha = expf(log_decay(ld_in(z + tid), escale, a.g_min));
        }
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

    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f), pb = pa;
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int c = row0 + m * RPP;
        const float ak = s_ak[c], aq = s_aq[c];
        pa.x = fmaf(ak, st[m].x, pa.x); pa.y = fmaf(ak, st[m].y, pa.y);
        pa.z = fmaf(ak, st[m].z, pa.z); pa.w = fmaf(ak, st[m].w, pa.w);
        pb.x = fmaf(aq, st[m].x, pb.x); pb.y = fmaf(aq, st[m].y, pb.y);
        pb.z = fmaf(aq, st[m].z, pb.z); pb.w = fmaf(aq, st[m].w, pb.w);
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
        st_out(o + tid, a.scale * fmaf(kq, u, bv));
    }
    __syncthreads();

    const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[col4 * 4]);
#pragma unroll
    for (int m = 0; m < PASSES; ++m) {
        const int c = row0 + m * RPP;
        const float al = s_alpha[c], kc = s_k[c];
        float4 r;
        r.x = fmaf(al, st[m].x, kc * u4.x); r.y = fmaf(al, st[m].y, kc * u4.y);
        r.z = fmaf(al, st[m].z, kc * u4.z); r.w = fmaf(al, st[m].w, kc * u4.w);
        st_stream(S + c * V4 + col4, r);
    }
}

template <int DK, int DVS>
struct DecodeSmem {
    float2 akq[kTokBlock][DK];         // (alpha k, alpha q) per token and channel
    float2 alk[kTokBlock][DK];         // (alpha, k)
    float red[2][kDecodeThreads / (DVS / 4)][DVS];    // [a|b][row group][slab column]
    float4 u[DVS / 4];
    float v[kTokBlock][DVS];
    float kq[kTokBlock][DK / 32];      // per-warp partial sums of k.q
    float beta[kTokBlock];
};

// State load that the compiler may neither drop nor move below a branch:
// the loads are issued before the accepted count is known.
__device__ __forceinline__ float4 ld_state(const float4 *p) {
    float4 v;
    asm volatile("ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// Multi-token replay.  The value columns of the state never interact, so a
// (sequence, head) is split into CS slabs of DV / CS columns, one CTA each:
// half the registers per thread, so four CTAs share an SM and one CTA's
// state streaming overlaps another's token arithmetic.  Inside a slab, the
// single step's row layout: RPP row groups x V4 float4 columns; thread
// (rg, c4) holds rows rg + m RPP of slab column c4.  Per token: in-thread
// partial sums over its rows; barrier; the slab's threads add the RPP
// partials of one column each, form u_j and o_j; barrier; every thread
// applies u to its rows.  The second barrier also orders the partials'
// reads before the next token's writes, so one buffer serves all tokens.
// GenericGate = false compiles the default gate (eq. (5), one input per key
// channel) with the gate-mode tests and the staging loop's chunk count
// constant; true takes any kda_gate_mode.
template <typename Tin, int DK, int DV, int CS, bool GenericGate>
__global__ void __launch_bounds__(kDecodeThreads, 2 * CS) decode_kernel(DecodeArgs a) {
    constexpr int DVS = DV / CS;                     // slab columns
    constexpr int V4 = DVS / 4;                      // float4 per slab row
    constexpr int RPP = kDecodeThreads / V4;         // row groups
    constexpr int RPL = DK / RPP;                    // rows per thread
    static_assert(RPL >= 1 && DK % RPP == 0, "tiling");

    __shared__ __align__(16) DecodeSmem<DK, DVS> sm;

    const int tid = threadIdx.x, lane = tid & 31;
    const int c4 = tid % V4, rg = tid / V4;
    const int nh = blockIdx.x / CS;                  // n * H + h
    const int slab = blockIdx.x % CS;
    const int n = nh / a.H, h = nh % a.H;

    const int acc_raw = a.accepted ? __ldg(a.accepted + n) : a.K;
    // Issue the state loads first: they dominate the kernel's time.
    float4 *S = reinterpret_cast<float4 *>(a.state) + static_cast<size_t>(nh) * (DK * (DV / 4)) + slab * V4;
    f32x2 st[RPL][2];
#pragma unroll
    for (int m = 0; m < RPL; ++m) {
        const float4 x = ld_state(S + (rg + m * RPP) * (DV / 4) + c4);
        st[m][0] = pack2(x.x, x.y);
        st[m][1] = pack2(x.z, x.w);
    }

    const float escale = a.A_log ? expf(__ldg(a.A_log + h)) : 1.0f;
    const size_t tok_k = static_cast<size_t>(a.H) * DK, tok_v = static_cast<size_t>(a.H) * DV;
    const Tin *gq = static_cast<const Tin *>(a.q);
    const Tin *gk = static_cast<const Tin *>(a.k);
    const Tin *gz = static_cast<const Tin *>(a.g);
    const Tin *gv = static_cast<const Tin *>(a.v);
    const Tin *gb = static_cast<const Tin *>(a.beta);
    Tin *go = static_cast<Tin *>(a.out);

    // bf16 drafts: the block's q, k, g_raw rows and v slab rows are copied into
    // shared memory (over the reduction buffer, idle until the token loop) by
    // 16-byte asynchronous copies, all in flight at once.
    constexpr bool kStage = sizeof(Tin) == 2;
    static_assert(!kStage || sizeof(sm.red) >= (3 * kTokBlock * DK + kTokBlock * DVS) * sizeof(Tin), "staging");
    Tin *kin = reinterpret_cast<Tin *>(&sm.red[0][0][0]);
    Tin *qin = kin + kTokBlock * DK, *zin = qin + kTokBlock * DK, *vin = zin + kTokBlock * DK;
    auto stage = [&](int i0, int nb) {
        constexpr int CH = DK * static_cast<int>(sizeof(Tin)) / 16;    // 16-byte chunks per channel row
        constexpr int CV = DVS * static_cast<int>(sizeof(Tin)) / 16;   // per value-slab row
        const int nz = !GenericGate || (a.gate_mode != KDA_GATE_NONE && !a.gate_scalar) ? 1 : 0;
        const int per_tok = CH * (2 + nz) + CV;
        for (int idx = tid; idx < nb * per_tok; idx += kDecodeThreads) {
            const int i = idx / per_tok, w = idx % per_tok;
            const size_t tok = static_cast<size_t>(n) * a.K + i0 + i;
            if (w < CH * (2 + nz)) {
                const int m = w / CH, ch = w % CH;
                const Tin *src = (m == 0 ? gk : (m == 1 ? gq : gz)) + tok * tok_k + static_cast<size_t>(h) * DK;
                Tin *dst = (m == 0 ? kin : (m == 1 ? qin : zin)) + i * DK;
                cp_async16(dst + ch * (16 / sizeof(Tin)), src + ch * (16 / sizeof(Tin)));
            } else {
                const int ch = w - CH * (2 + nz);
                cp_async16(vin + i * DVS + ch * (16 / sizeof(Tin)),
                           gv + tok * tok_v + static_cast<size_t>(h) * DV + slab * DVS + ch * (16 / sizeof(Tin)));
            }
        }
        cp_async_wait_all();
        __syncthreads();
    };
    // Per-token vectors of tokens [i0, i0 + nb) (a warp's 32 channels share a token).
    auto prepare = [&](int i0, int nb) {
#pragma unroll 1
        for (int idx = tid; idx < nb * DK; idx += kDecodeThreads) {
            const int i = idx / DK, c = idx % DK;
            float kc, qc, zc;
            if constexpr (kStage) {
                kc = __bfloat162float(kin[i * DK + c]);
                qc = __bfloat162float(qin[i * DK + c]);
                zc = !GenericGate ? __bfloat162float(zin[i * DK + c])
                     : a.gate_mode == KDA_GATE_NONE ? 0.f
                     : a.gate_scalar ? ld_in(gz + (static_cast<size_t>(n) * a.K + i0 + i) * a.H + h)
                                     : __bfloat162float(zin[i * DK + c]);
            } else {
                const size_t o = (static_cast<size_t>(n) * a.K + i0 + i) * tok_k + static_cast<size_t>(h) * DK + c;
                kc = ld_in(gk + o);
                qc = ld_in(gq + o);
                const size_t og = GenericGate && a.gate_scalar ? (static_cast<size_t>(n) * a.K + i0 + i) * a.H + h : o;
                zc = GenericGate && a.gate_mode == KDA_GATE_NONE ? 0.f : ld_in(gz + og);
            }
            // the default gate on the MUFU path (as the tensor-core prefill):
            // alpha = 2^(log2(e) g_min / (1 + 2^(-log2(e) e^A z)))
            const float alpha =
                GenericGate ? expf(gate_log_decay(a.gate_mode, zc, escale, a.g_min))
                            : tcu::ex2_approx(tcu::kLog2e * a.g_min *
                                              tcu::rcp_approx(1.f + tcu::ex2_approx(-tcu::kLog2e * escale * zc)));
            sm.akq[i][c] = make_float2(alpha * kc, alpha * qc);
            sm.alk[i][c] = make_float2(alpha, kc);
            float kq = kc * qc;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if (lane == 0) sm.kq[i][c / 32] = kq;
        }
        for (int idx = tid; idx < nb * DVS; idx += kDecodeThreads) {
            if constexpr (kStage) {
                sm.v[idx / DVS][idx % DVS] = __bfloat162float(vin[idx]);
            } else {
                sm.v[idx / DVS][idx % DVS] =
                    ld_in(gv + (static_cast<size_t>(n) * a.K + i0 + idx / DVS) * tok_v + static_cast<size_t>(h) * DV +
                          slab * DVS + idx % DVS);
            }
        }
        if (tid < nb) sm.beta[tid] = ld_in(gb + (static_cast<size_t>(n) * a.K + i0 + tid) * a.H + h);
    };
    // The accepted count is read first; the first block's accepted drafts are
    // staged while the state's loads are in flight, and the vectors are
    // prepared for the accepted tokens only.
    const int n_acc = min(max(acc_raw, 0), a.K);
    if constexpr (kStage) {
        if (n_acc == 0) return;                      // state and outputs untouched
        stage(0, min(kTokBlock, n_acc));
        prepare(0, min(kTokBlock, n_acc));
    } else {
        prepare(0, min(kTokBlock, a.K));
        if (n_acc == 0) return;
    }
    __syncthreads();

#pragma unroll 1
    for (int i0 = 0; i0 < n_acc; i0 += kTokBlock) {
        const int nb = min(kTokBlock, n_acc - i0);
        if (i0 > 0) {
            __syncthreads();                         // previous block's vectors are consumed
            if constexpr (kStage) stage(i0, nb);
            prepare(i0, nb);
            __syncthreads();
        }
#pragma unroll 1
        for (int i = 0; i < nb; ++i) {
            // partial a_j = sum_c alpha_c k_c S_cj and b_j = sum_c alpha_c q_c S_cj over this thread's rows
            f32x2 pa0 = 0ull, pa1 = 0ull, pb0 = 0ull, pb1 = 0ull;     // +0.0f in both lanes
#pragma unroll
            for (int m = 0; m < RPL; ++m) {   // one 8-byte load per row; the pairs are built in registers
                const float2 ch = sm.akq[i][rg + m * RPP];
                const f32x2 ak = pack2(ch.x, ch.x), aq = pack2(ch.y, ch.y);
                pa0 = ffma2(ak, st[m][0], pa0); pa1 = ffma2(ak, st[m][1], pa1);
                pb0 = ffma2(aq, st[m][0], pb0); pb1 = ffma2(aq, st[m][1], pb1);
            }
            {
                const float2 a0 = unpack2(pa0), a1 = unpack2(pa1), b0 = unpack2(pb0), b1 = unpack2(pb1);
                *reinterpret_cast<float4 *>(&sm.red[0][rg][4 * c4]) = make_float4(a0.x, a0.y, a1.x, a1.y);
                *reinterpret_cast<float4 *>(&sm.red[1][rg][4 * c4]) = make_float4(b0.x, b0.y, b1.x, b1.y);
            }
            __syncthreads();
            if (tid < DVS) {
                float av = 0.f, bv = 0.f;
#pragma unroll
                for (int r = 0; r < RPP; ++r) {
                    av += sm.red[0][r][tid];
                    bv += sm.red[1][r][tid];
                }
                float kq = 0.f;
#pragma unroll
                for (int w = 0; w < DK / 32; ++w) kq += sm.kq[i][w];
                const float u = sm.beta[i] * (sm.v[i][tid] - av);
                reinterpret_cast<float *>(sm.u)[tid] = u;
                st_out(go + (static_cast<size_t>(n) * a.K + i0 + i) * tok_v + static_cast<size_t>(h) * DV +
                           slab * DVS + tid,
                       a.scale * fmaf(kq, u, bv));
            }
            __syncthreads();
            // S = Diag(alpha) S + k u^T
            const float4 u = sm.u[c4];
            const f32x2 u0 = pack2(u.x, u.y), u1 = pack2(u.z, u.w);
#pragma unroll
            for (int m = 0; m < RPL; ++m) {
                const float2 ch = sm.alk[i][rg + m * RPP];
                const f32x2 al = pack2(ch.x, ch.x), kk = pack2(ch.y, ch.y);
                st[m][0] = ffma2(al, st[m][0], fmul2(kk, u0));
                st[m][1] = ffma2(al, st[m][1], fmul2(kk, u1));
            }
        }
    }
#pragma unroll
    for (int m = 0; m < RPL; ++m) {
        const float2 x = unpack2(st[m][0]), y = unpack2(st[m][1]);
        st_stream(S + (rg + m * RPP) * (DV / 4) + c4, make_float4(x.x, x.y, y.x, y.y));
    }
}

template <typename Tin>
cudaError_t launch_t(int dk, int dv, const DecodeArgs &a, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>(a.N) * static_cast<unsigned>(a.H));
    const dim3 block(kDecodeThreads);
    const bool single = a.K == 1 && !a.accepted;
    const bool default_gate = a.gate_mode == KDA_GATE_BOUNDED && !a.gate_scalar;
#define KDA_DEC_CASE(DK_, DV_)                                            \
    if (dk == DK_ && dv == DV_) {                                         \
        if (single && default_gate)                                       \
            decode1_kernel<Tin, DK_, DV_, false><<<grid, block, 0, s>>>(a); \
        else if (single) decode1_kernel<Tin, DK_, DV_, true><<<grid, block, 0, s>>>(a); \
        else if constexpr (DK_ == 128 && DV_ == 128) {                   \
            if (default_gate)                                             \
                decode_kernel<Tin, DK_, DV_, 2, false><<<dim3(grid.x * 2), block, 0, s>>>(a); \
            else decode_kernel<Tin, DK_, DV_, 2, true><<<dim3(grid.x * 2), block, 0, s>>>(a); \
        } else if constexpr (DV_ >= 64)                                   \
            decode_kernel<Tin, DK_, DV_, 2, true><<<dim3(grid.x * 2), block, 0, s>>>(a); \
        else decode_kernel<Tin, DK_, DV_, 1, true><<<grid, block, 0, s>>>(a); \
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
