// Segment split of the prefill: every sequence is cut into segments of
// seg_tokens tokens that run at the same time, and the exact result is
// assembled afterwards.
//
// Method: the recurrence of eq. (1) ("Kimi K3：从三条信息流到完整系统",
// §KDA 是带逐通道遗忘的 delta rule) is affine in the state it starts from.
// Over a segment starting from S_in,
//     S_t = Phi_t S_in + S0_t,      o_t = o0_t + S_in^T (Phi_t^T q_t),
// where (S0, o0) is the segment run from a zero state and Phi_t (dk x dk) is
// the segment run with v = 0 from S = I: its state is Phi_t and its output
// Phi_t^T q_t.  The pages compose segments exactly this way across devices
// (§FlashKDA 与 KCP, eq. (17): a segment is the pair (M, E) = (Phi, S0) and
// consecutive pairs compose as (M2 M1, M2 E1 + E2)) and across the
// multiprocessors of one chip ("Kimi K3: Two point eight trillion
// parameters, open weights, and forty-seven pages of how", §The machine
// underneath).  Here one launch of the tensor-core prefill runs, for every
// sequence, segment 0 from its given initial state, segments 1.. from zero,
// and the transition run of each segment 1.., every run writing its output
// rows unrounded (fp32; one output path, so the runs' tile loop carries no
// per-run branch); then
//   split_compose_kernel: S_in,1 = final state of segment 0 and
//       S_in,p+1 = Phi_p S_in,p + S0_p (fp32), the last one the final state;
//   split_fixup_kernel:   o_t = o0_t + S_in,p^T R_t for t in segment p >= 1,
//       R the transition run's output rows, the product on fp16 copies with
//       fp32 sums, and o_t = o0_t in segment 0; o_t is rounded to bf16 once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kda_internal.cuh"
#include "kda_tc_util.cuh"

namespace kda {
namespace {
using namespace tcu;

constexpr int D = 128;

// Sequence n's token span, clamped like the prefill's.
__device__ __forceinline__ void span_of(const SplitArgs &a, int n, int &b, int &e) {
    if (a.cu_seqlens) {
        b = min(max(a.cu_seqlens[n], 0), a.T_total);
        e = min(max(a.cu_seqlens[n + 1], b), a.T_total);
    } else {
        b = n * a.T_seq;
        e = b + a.T_seq;
    }
}
__device__ __forceinline__ int segments_of(const SplitArgs &a, int n) {
    int b, e;
    span_of(a, n, b, e);
    return max(1, (e - b + a.seg_tokens - 1) / a.seg_tokens);
}

// One CTA of 1024 threads.  Sequence n with P segments owns the 2P - 1
// virtual sequences from base_n = sum over m < n of (2 P_m - 1): base_n + p
// runs segment p (p = 0: the given initial state; p >= 1: zero), and
// base_n + P + p - 1 the transition run of segment p >= 1, whose .w holds
// base_n + p, the slot of the state entering that segment.  Entries past
// the total are empty.
__global__ void __launch_bounds__(1024) split_plan_kernel(SplitArgs a) {
    __shared__ int warp_sums[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (a.N + 1023) / 1024;
    const int n0 = min(tid * per, a.N), n1 = min(n0 + per, a.N);
    int mine = 0;
    for (int n = n0; n < n1; ++n) mine += 2 * segments_of(a, n) - 1;
    // exclusive scan of `mine` over the block
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane], wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        warp_sums[lane] = wi - w;   // exclusive prefix of the warps
    }
    __syncthreads();
    int base = warp_sums[warp] + incl - mine;
    for (int n = n0; n < n1; ++n) {
        int b, e;
        span_of(a, n, b, e);
        const int P = max(1, (e - b + a.seg_tokens - 1) / a.seg_tokens);
        a.seqtab[n] = make_int2(base, P);
        for (int p = 0; p < P; ++p) {
            const int sb = min(b + p * a.seg_tokens, e), se = min(sb + a.seg_tokens, e);
            if (base + p < a.nv_max)
                a.vseg[base + p] = make_int4(sb, se, p == 0 ? VSEG_OUT_ZERO | VSEG_OUT_FINAL
                                                            : VSEG_ZERO_INIT | VSEG_OUT_ZERO, n);
            if (p > 0 && base + P + p - 1 < a.nv_max)
                a.vseg[base + P + p - 1] =
                    make_int4(sb, se, VSEG_ZERO_V | VSEG_IDENT_INIT | VSEG_OUT_TRANS, base + p);
        }
        base += 2 * P - 1;
    }
    // the block's total: the last thread's inclusive end
    __shared__ int total;
    if (tid == 1023) total = base;
    __syncthreads();
    for (int i = total + tid; i < a.nv_max; i += 1024) a.vseg[i] = make_int4(0, 0, VSEG_EMPTY, 0);
}

// State composition over one (sequence, head), CW of the state's columns
// per CTA (blockIdx.y picks them): S = s_first, then for p = 1 .. P - 1:
// keep_of(p) <- S (the state entering segment p, when the pointer is set),
// S <- phi_of(p) S + s0_of(p); final <- S (when set).  The columns of S
// never mix (each is advanced by the same Phi), so the column blocks of one
// chain run on separate CTAs with no exchange.  256 threads, each 8 rows of
// one column; shared memory: Phi^T (row stride CPAD) and the CTA's columns
// of S.  Phi of the next step is loaded into registers while the current
// product runs.
constexpr int CPAD = 132;
constexpr int CW = 16;
constexpr int COMPOSE_SMEM = (D * CPAD + D * CW) * 4;

template <typename PhiOf, typename S0Of, typename KeepOf>
__device__ __forceinline__ void compose_chain(float *csm, int P, const float *s_first, PhiOf phi_of, S0Of s0_of,
                                              KeepOf keep_of, float *final_out) {
    float *phiT = csm;              // phiT[c][r] = Phi[r][c]
    float *sc = csm + D * CPAD;     // sc[c][jj] = S[c][jb + jj]
    const int tid = threadIdx.x, jb = static_cast<int>(blockIdx.y) * CW;
    const int r0 = (tid >> 4) * 8, jj = tid & (CW - 1);
    static_assert(CW == 16 && D == 128, "thread layout: 16 row groups x 16 columns");
    // this CTA's columns of a [D, D] state as float4 chunks i: row i / (CW / 4), columns 4 (i % (CW / 4)) ..
    auto cols4 = [&](const float *m, int i) {
        return reinterpret_cast<const float4 *>(m + (i / (CW / 4)) * D + jb) + (i % (CW / 4));
    };
    for (int i = tid; i < D * CW / 4; i += 256) reinterpret_cast<float4 *>(sc)[i] = *cols4(s_first, i);
    // Phi as 16 float4 per thread: chunk i = tid + 256 k is row i & 127,
    // columns 4 (i >> 7) .., so a warp's lanes hold 32 consecutive rows and
    // its transposed stores fall in 32 distinct banks
    float4 x[16];
    auto load_phi = [&](int p) {
        const float4 *phi = reinterpret_cast<const float4 *>(phi_of(p));
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int i = tid + 256 * k;
            x[k] = phi[(i & 127) * (D / 4) + (i >> 7)];
        }
    };
    if (P > 1) load_phi(1);
    __syncthreads();
    for (int p = 1; p < P; ++p) {
        if (float *keep = keep_of(p))
            for (int i = tid; i < D * CW / 4; i += 256)
                *const_cast<float4 *>(cols4(keep, i)) = reinterpret_cast<const float4 *>(sc)[i];
        const float *s0 = s0_of(p);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = s0[(r0 + i) * D + jb + jj];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int i = tid + 256 * k, r = i & 127, c = (i >> 7) * 4;
            phiT[(c + 0) * CPAD + r] = x[k].x;
            phiT[(c + 1) * CPAD + r] = x[k].y;
            phiT[(c + 2) * CPAD + r] = x[k].z;
            phiT[(c + 3) * CPAD + r] = x[k].w;
        }
        __syncthreads();
        if (p + 1 < P) load_phi(p + 1);   // in flight during the product
#pragma unroll 4
        for (int c = 0; c < D; ++c) {
            const float4 pa = *reinterpret_cast<const float4 *>(phiT + c * CPAD + r0);
            const float4 pb = *reinterpret_cast<const float4 *>(phiT + c * CPAD + r0 + 4);
            const float sv = sc[c * CW + jj];
            acc[0] = fmaf(pa.x, sv, acc[0]); acc[1] = fmaf(pa.y, sv, acc[1]);
            acc[2] = fmaf(pa.z, sv, acc[2]); acc[3] = fmaf(pa.w, sv, acc[3]);
            acc[4] = fmaf(pb.x, sv, acc[4]); acc[5] = fmaf(pb.y, sv, acc[5]);
            acc[6] = fmaf(pb.z, sv, acc[6]); acc[7] = fmaf(pb.w, sv, acc[7]);
        }
        __syncthreads();   // every thread has read S and Phi^T
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[(r0 + i) * CW + jj] = acc[i];
        __syncthreads();
    }
    if (final_out)
        for (int i = tid; i < D * CW / 4; i += 256)
            *const_cast<float4 *>(cols4(final_out, i)) = reinterpret_cast<const float4 *>(sc)[i];
}

__global__ void __launch_bounds__(256) split_compose_kernel(SplitArgs a) {
    extern __shared__ float csm[];
    const int n = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const int2 st = a.seqtab[n];
    const int base = st.x, P = st.y;
    const size_t hs = static_cast<size_t>(D) * D;
    auto slot = [&](float *buf, int v) { return buf + (static_cast<size_t>(v) * a.H + h) * hs; };
    // segment p's run from zero is virtual sequence base + p, its transition
    // run base + P + p - 1; segment 0's run (from the given state) ends in
    // the state entering segment 1
    compose_chain(csm, P, slot(a.states, base), [&](int p) { return slot(a.states, base + P + p - 1); },
                  [&](int p) { return slot(a.states, base + p); }, [&](int p) { return slot(a.s_in, base + p); },
                  a.final_state ? a.final_state + (static_cast<size_t>(n) * a.H + h) * hs : nullptr);
}

// o_t = o0_t + S_in^T R_t over tokens [t_first, t_end) of head h: 64 rows at
// a time.  S_in (fp32) is held as fp16 B fragments in shared memory, laid out
// [j][c] (row stride 136 halves, conflict-free); R (fp32) is staged as fp16
// [t][c] (same stride), the next 64 rows loaded into registers while the
// current ones are multiplied.  Warp w computes rows 16 (w & 3) .. +16 and
// columns 64 (w >> 2) .. +64 of the 64 x 128 update with m16n8k16 fp16
// products.  Rows are [token][H][128] in R, O0 and O.
constexpr int FIX_TOKENS = 1024;
constexpr int HSTR = 136;                         // fp16 row stride of S_in^T (bank spread)
constexpr int FT = 32;                            // tokens per stage
constexpr int RPAD = 136;                         // fp32 row stride of the staged rows
constexpr int FIX_STAGE = 2 * FT * RPAD * 4;      // R and o0 rows of one stage
constexpr int FIX_SMEM = D * HSTR * 2 + 2 * FIX_STAGE;

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// o_t = bf16(o0_t + S_in^T R_t) for the tokens [t_first, t_end) of head h.
// R and o0 rows stream through two shared-memory stages of FT tokens by
// 16-byte cp.async (no registers held while in flight; stage k + 1 loads
// while stage k is used); S_in^T is converted to fp16 once.  Eight warps,
// warp w the rows 16 (w & 1) .. and columns 32 (w >> 1) .. of a stage's
// [FT, 128] output: m16n8k16 products, A (R rows) converted from fp32 in
// registers, fp32 sums, one bf16 rounding.
__device__ __forceinline__ void fixup_span(unsigned char *fsm, int t_first, int t_end, int h, int H,
                                           const float *sin_, const float *R, const float *O0,
                                           __nv_bfloat16 *O) {
    __half *sT = reinterpret_cast<__half *>(fsm);                 // sT[j][c] = S_in[c][j]
    float *stage0 = reinterpret_cast<float *>(fsm + D * HSTR * 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // stage buf: rows [t0, t0 + FT) of R then of o0, RPAD floats a row;
    // 2 x FT x 32 chunks of 16 bytes, 8 a thread; rows past t_end are not
    // loaded (their products are never stored); one commit group a stage
    auto load_stage = [&](int t0, int buf) {
        float *st = stage0 + buf * (2 * FT * RPAD);
#pragma unroll
        for (int k = 0; k < 2 * FT * 32 / 256; ++k) {
            const int i = tid + 256 * k;
            const int which = i / (FT * 32), row = (i / 32) % FT, ch = i % 32;
            const int t = t0 + row;
            if (t < t_end)
                cp_async16(st + (which * FT + row) * RPAD + ch * 4,
                           (which ? O0 : R) + (static_cast<size_t>(t) * H + h) * D + ch * 4);
        }
        cp_async_commit();
    };
    load_stage(t_first, 0);
    {   // S_in^T as fp16: thread tid converts float4 chunks (row c, columns 4 m ..)
        float4 x[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) x[k] = reinterpret_cast<const float4 *>(sin_)[tid + 256 * k];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int i = tid + 256 * k, c = i >> 5, j0 = (i & 31) * 4;
            sT[(j0 + 0) * HSTR + c] = __float2half_rn(x[k].x);
            sT[(j0 + 1) * HSTR + c] = __float2half_rn(x[k].y);
            sT[(j0 + 2) * HSTR + c] = __float2half_rn(x[k].z);
            sT[(j0 + 3) * HSTR + c] = __float2half_rn(x[k].w);
        }
    }
    const int g = lane >> 2, tq = lane & 3;
    constexpr int NB = 4;                          // n8 blocks a warp
    const int m0 = 16 * (warp & 1), n0 = 32 * (warp >> 1);
    int buf = 0;
    for (int t0 = t_first; t0 < t_end; t0 += FT, buf ^= 1) {
        load_stage(t0 + FT, buf ^ 1);              // an empty group past t_end
        cp_async_wait<1>();                        // this thread's copies of stage buf are done
        __syncthreads();                           // everyone's; S_in^T written (first pass)
        const float *rs = stage0 + buf * (2 * FT * RPAD);
        const float *os = rs + FT * RPAD;
        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[nb][q] = 0.f;
#pragma unroll
        for (int k0 = 0; k0 < D; k0 += 16) {
            const float2 x0 = *reinterpret_cast<const float2 *>(rs + (m0 + g) * RPAD + k0 + 2 * tq);
            const float2 x1 = *reinterpret_cast<const float2 *>(rs + (m0 + g + 8) * RPAD + k0 + 2 * tq);
            const float2 x2 = *reinterpret_cast<const float2 *>(rs + (m0 + g) * RPAD + k0 + 2 * tq + 8);
            const float2 x3 = *reinterpret_cast<const float2 *>(rs + (m0 + g + 8) * RPAD + k0 + 2 * tq + 8);
            const uint32_t a0 = pack_h2(x0.x, x0.y), a1 = pack_h2(x1.x, x1.y);
            const uint32_t a2 = pack_h2(x2.x, x2.y), a3 = pack_h2(x3.x, x3.y);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int j = n0 + 8 * nb + g;
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(sT + j * HSTR + k0 + 2 * tq);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(sT + j * HSTR + k0 + 2 * tq + 8);
                mma_16816_f16(acc[nb], a0, a1, a2, a3, b0, b1);
            }
        }
        // rows m0 + g (acc[.][0..1]) and m0 + g + 8 (acc[.][2..3]), columns n0 + 8 nb + 2 tq + {0, 1}
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int r = m0 + g + 8 * hr, t = t0 + r;
            if (t >= t_end) continue;
            __nv_bfloat16 *orow = O + (static_cast<size_t>(t) * H + h) * D;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int col = n0 + 8 * nb + 2 * tq;
                const float2 o0 = *reinterpret_cast<const float2 *>(os + r * RPAD + col);
                *reinterpret_cast<__nv_bfloat162 *>(orow + col) =
                    __floats2bfloat162_rn(o0.x + acc[nb][2 * hr], o0.y + acc[nb][2 * hr + 1]);
            }
        }
        __syncthreads();                           // stage buf consumed before it is refilled
    }
    cp_async_wait<0>();
}

// o_t = bf16(O0_t) for the tokens [t_first, t_end) of head h (a first
// segment, whose run started from the sequence's own initial state): float4
// chunks (row i / 32, channels 4 (i % 32) ..), four loads in flight a thread.
__device__ __forceinline__ void round_span(int t_first, int t_end, int h, int H, const float *O0,
                                           __nv_bfloat16 *O) {
    const int n4 = (t_end - t_first) * (D / 4);
    for (int i0 = threadIdx.x; i0 < n4; i0 += 4 * 256) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + 256 * u;
            if (i < n4)
                x[u] = *reinterpret_cast<const float4 *>(
                    O0 + (static_cast<size_t>(t_first + i / (D / 4)) * H + h) * D + 4 * (i % (D / 4)));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + 256 * u;
            if (i < n4) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(x[u].x, x[u].y), hi = __floats2bfloat162_rn(x[u].z, x[u].w);
                uint2 w;
                w.x = *reinterpret_cast<uint32_t *>(&lo);
                w.y = *reinterpret_cast<uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(O + (static_cast<size_t>(t_first + i / (D / 4)) * H + h) * D +
                                           4 * (i % (D / 4))) = w;
            }
        }
    }
}

// CTA (virtual index, chunk, head): FIX_TOKENS tokens of a transition run's
// segment (corrected), or of a first segment (rounded).
__global__ void __launch_bounds__(256) split_fixup_kernel(SplitArgs a) {
    extern __shared__ __align__(16) unsigned char fsm[];
    const int vi = blockIdx.x, h = blockIdx.z;
    const int4 e = a.vseg[vi];
    if (!(e.z & (VSEG_OUT_TRANS | VSEG_OUT_FINAL))) return;   // one CTA row per transition run or first segment
    const int t_first = e.x + blockIdx.y * FIX_TOKENS;
    const int t_end = min(e.y, t_first + FIX_TOKENS);
    if (t_first >= t_end) return;
    if (e.z & VSEG_OUT_FINAL) {
        round_span(t_first, t_end, h, a.H, a.out_zero, static_cast<__nv_bfloat16 *>(a.out));
        return;
    }
    fixup_span(fsm, t_first, t_end, h, a.H, a.s_in + (static_cast<size_t>(e.w) * a.H + h) * D * D, a.out_trans,
               a.out_zero, static_cast<__nv_bfloat16 *>(a.out));
}

// Sequence split across ranks (KCP): rank r >= 1 holds tokens of B
// sequences of T tokens each; for each it runs the zero-state run (virtual
// 2n) and the transition run (2n + 1) over its tokens.
__global__ void __launch_bounds__(256) kcp_plan_kernel(KcpArgs a) {
    for (int n = threadIdx.x; n < a.B; n += 256) {
        a.vseg[2 * n] = make_int4(n * a.T, (n + 1) * a.T, VSEG_ZERO_INIT | VSEG_OUT_ZERO, n);
        a.vseg[2 * n + 1] = make_int4(n * a.T, (n + 1) * a.T, VSEG_ZERO_V | VSEG_IDENT_INIT | VSEG_OUT_TRANS, n);
    }
}

// One CTA per (sequence, head, column block): the state entering rank r from the gathered
// pairs of ranks 0 .. r ([r + 1, B, 2, H, d, d]: [.][.][0] the zero-state
// run's final state (rank 0: its true final state), [.][.][1] the
// transition), then this rank's final state.
__global__ void __launch_bounds__(256) kcp_compose_kernel(KcpArgs a) {
    extern __shared__ float csm[];
    const int n = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const size_t hs = static_cast<size_t>(D) * D;
    auto pair = [&](int rank, int which) {
        return a.pairs + ((((static_cast<size_t>(rank) * a.B + n) * 2 + which) * a.H) + h) * hs;
    };
    float *keep = a.s_in + (static_cast<size_t>(n) * a.H + h) * hs;
    compose_chain(csm, a.rank + 1, pair(0, 0), [&](int p) { return pair(p, 1); }, [&](int p) { return pair(p, 0); },
                  [&](int p) { return p == a.rank ? keep : static_cast<float *>(nullptr); },
                  a.final_state ? a.final_state + (static_cast<size_t>(n) * a.H + h) * hs : nullptr);
}

// CTA (sequence, chunk, head): FIX_TOKENS tokens of this rank's part of a sequence.
__global__ void __launch_bounds__(256) kcp_fixup_kernel(KcpArgs a) {
    extern __shared__ __align__(16) unsigned char fsm[];
    const int n = blockIdx.x, h = blockIdx.z;
    const int t_first = n * a.T + blockIdx.y * FIX_TOKENS;
    const int t_end = min((n + 1) * a.T, t_first + FIX_TOKENS);
    if (t_first >= t_end) return;
    fixup_span(fsm, t_first, t_end, h, a.H, a.s_in + (static_cast<size_t>(n) * a.H + h) * D * D, a.out_trans,
               a.out_zero, static_cast<__nv_bfloat16 *>(a.out));
}

}  // namespace

cudaError_t launch_kcp_plan(const KcpArgs &a, cudaStream_t s) {
    kcp_plan_kernel<<<1, 256, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t launch_kcp_finish(const KcpArgs &a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kcp_compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         COMPOSE_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kcp_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FIX_SMEM);
    if (e != cudaSuccess) return e;
    kcp_compose_kernel<<<dim3(static_cast<unsigned>(a.B) * static_cast<unsigned>(a.H), D / CW), 256, COMPOSE_SMEM,
                         s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    const dim3 grid(static_cast<unsigned>(a.B), static_cast<unsigned>((a.T + FIX_TOKENS - 1) / FIX_TOKENS),
                    static_cast<unsigned>(a.H));
    kcp_fixup_kernel<<<grid, 256, FIX_SMEM, s>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t launch_split_plan(const SplitArgs &a, cudaStream_t s) {
    split_plan_kernel<<<1, 1024, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t launch_split_compose(const SplitArgs &a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(split_compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         COMPOSE_SMEM);
    if (e != cudaSuccess) return e;
    split_compose_kernel<<<dim3(static_cast<unsigned>(a.N) * static_cast<unsigned>(a.H), D / CW), 256, COMPOSE_SMEM,
                           s>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t launch_split_fixup(const SplitArgs &a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(split_fixup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FIX_SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(a.nv_max), static_cast<unsigned>((a.seg_tokens + FIX_TOKENS - 1) / FIX_TOKENS),
                    static_cast<unsigned>(a.H));
    split_fixup_kernel<<<grid, 256, FIX_SMEM, s>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace kda
