// The passes on either side of the KDA operator ("Kimi K3：从三条信息流到完整系统",
// §从投影到 Chunkwise 的完整接口, eq. (2), and §下界 log-decay 是一个 kernel 设计,
// eq. (6)):
//
//   prep : q, k = L2Norm(Swish(ShortConv(x_q|k))),  v = Swish(ShortConv(x_v)),
//          beta = Sigmoid(beta_logit)
//   post : y = Sigmoid(gate) * RMSNorm(o)            (before the W_o projection)
//
// The projections W x themselves are plain GEMMs and stay outside.  ShortConv
// is the causal depthwise convolution of kernel size 4 along the tokens of
// each sequence (the model's short_conv_kernel_size):
//   y_t[ch] = sum_{i=0..3} w[ch][i] * x_{t-3+i}[ch],
// with x before a sequence's first token taken from the caller's conv state
// (the last three inputs of the previous call) or zero.  L2Norm divides each
// head's d channels by sqrt(sum x^2 + eps); RMSNorm divides by
// sqrt(mean x^2 + eps) and multiplies by a per-channel weight shared by the
// heads.
//
// Both passes are HBM-bound streams.  prep: one CTA owns two consecutive
// runs of 64 tokens of one (tensor, head): a TMA copy per run brings it and
// the three tokens before it ([67, d], rows before the first token read as
// zero) into shared memory, both requested up front, so many runs are in
// flight per SM without holding registers; in each of four warps a group of d/8 lanes owns a
// token (8 channels per lane, 16-byte loads and stores) and walks its
// share of the warp's 16 tokens with the three previous inputs in
// registers, the L2 norm as a group reduction.  A run that stays inside one
// sequence takes straight-line code; inputs before a sequence's first token
// come from the caller's conv state (or zero), never from the previous
// sequence.
// post: one warp per (token, head) row, four rows per warp in flight.
#include <type_traits>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

constexpr int kRun = 64;          // tokens per prep CTA
constexpr int kHalo = 3;          // inputs before the run that ShortConv reads
constexpr int kPrepWarps = 4;     // prep warps, kRun / kPrepWarps tokens each
constexpr int kWarps = 8;         // warps per output-gate CTA
constexpr uint64_t kPrepWaitNs = 1000000000ull;   // bounded wait for the TMA tile (1 s)

__device__ unsigned int g_prep_timeouts = 0;

template <typename T, int CPL> struct Lanes;
template <> struct Lanes<__nv_bfloat16, 4> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&x)[4]) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(p));
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&w.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w.y);
        x[0] = __low2float(a); x[1] = __high2float(a); x[2] = __low2float(b); x[3] = __high2float(b);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&x)[4]) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t *>(&a);
        w.y = *reinterpret_cast<const uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = w;
    }
};
template <> struct Lanes<float, 4> {
    static __device__ __forceinline__ void load(const float *p, float (&x)[4]) {
        const float4 w = __ldg(reinterpret_cast<const float4 *>(p));
        x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
    }
    static __device__ __forceinline__ void store(float *p, const float (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};
// A lane's CPL channels of one token row in shared memory.
template <typename T, int CPL> struct LanesScalar {
    static __device__ __forceinline__ void load(const T *p, float (&x)[CPL]) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) x[i] = ld_in(p + i);
    }
    static __device__ __forceinline__ void store(T *p, const float (&x)[CPL]) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) st_out(p + i, x[i]);
    }
};
template <> struct Lanes<__nv_bfloat16, 2> : LanesScalar<__nv_bfloat16, 2> {};
template <> struct Lanes<__nv_bfloat16, 1> : LanesScalar<__nv_bfloat16, 1> {};
template <> struct Lanes<float, 2> : LanesScalar<float, 2> {};
template <> struct Lanes<float, 1> : LanesScalar<float, 1> {};

// Sigmoid from the hardware exponential and the fast division (relative
// error ~1e-7, far inside the outputs' rounding): the prep pass issues about
// 150 instructions per token and head, so the ~20 of an accurate expf and
// an IEEE division per element would bound it.  For x < -88, e^{-x}
// overflows and Sigmoid returns 0, its limit.
__device__ __forceinline__ float sigmoid(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// Swish of a channel pair: the exponentials and reciprocals stay per lane
// (MUFU), the rest is packed.  Same arithmetic as swish() per element.
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Sequence of token t: the n with cu[n] <= t < cu[n+1] (binary search over
// the clamped spans; empty sequences are skipped).
__device__ __forceinline__ int seq_of(const PrepArgs &a, int t) {
    if (!a.cu_seqlens) return t / a.T_seq;
    int lo = 0, hi = a.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (min(max(a.cu_seqlens[mid], 0), a.T_total) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}
__device__ __forceinline__ void span_of(const PrepArgs &a, int n, int &bos, int &eos) {
    if (a.cu_seqlens) {
        bos = min(max(a.cu_seqlens[n], 0), a.T_total);
        eos = min(max(a.cu_seqlens[n + 1], bos), a.T_total);
    } else {
        bos = n * a.T_seq;
        eos = bos + a.T_seq;
    }
}

template <typename Tin, int D>
__host__ __device__ constexpr int prep_tile_bytes() {
    return ((kRun + kHalo) * D * static_cast<int>(sizeof(Tin)) + 127) & ~127;
}
template <typename Tin, int D>
constexpr int prep_smem_bytes() {
    return 2 * prep_tile_bytes<Tin, D>() + D * 16 + 16;     // two run tiles + taps + two mbarriers
}

// Eight consecutive channels as four (even, odd) f32x2 pairs: global and
// shared-memory rows (16-byte aligned) of bf16 or fp32.
template <typename T> struct Oct;
template <> struct Oct<__nv_bfloat16> {
    static __device__ __forceinline__ void unpack(const uint4 w, sm100::f32x2 (&x)[4]) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) x[p] = sm100::pack2(__uint_as_float(u[p] << 16), __uint_as_float(u[p] & 0xffff0000u));
    }
    static __device__ __forceinline__ void ld_global(const __nv_bfloat16 *p, sm100::f32x2 (&x)[4]) {
        unpack(__ldg(reinterpret_cast<const uint4 *>(p)), x);
    }
    static __device__ __forceinline__ void ld_shared(const __nv_bfloat16 *p, sm100::f32x2 (&x)[4]) {
        unpack(*reinterpret_cast<const uint4 *>(p), x);
    }
    static __device__ __forceinline__ void st_global(__nv_bfloat16 *p, const sm100::f32x2 (&x)[4]) {
        uint32_t u[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = sm100::unpack2(x[q]);
            const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
            u[q] = *reinterpret_cast<const uint32_t *>(&b);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(u[0], u[1], u[2], u[3]);
    }
};
template <> struct Oct<float> {
    static __device__ __forceinline__ void from4(const float4 a, const float4 b, sm100::f32x2 (&x)[4]) {
        x[0] = sm100::pack2(a.x, a.y); x[1] = sm100::pack2(a.z, a.w);
        x[2] = sm100::pack2(b.x, b.y); x[3] = sm100::pack2(b.z, b.w);
    }
    static __device__ __forceinline__ void ld_global(const float *p, sm100::f32x2 (&x)[4]) {
        from4(__ldg(reinterpret_cast<const float4 *>(p)), __ldg(reinterpret_cast<const float4 *>(p) + 1), x);
    }
    static __device__ __forceinline__ void ld_shared(const float *p, sm100::f32x2 (&x)[4]) {
        from4(reinterpret_cast<const float4 *>(p)[0], reinterpret_cast<const float4 *>(p)[1], x);
    }
    static __device__ __forceinline__ void st_global(float *p, const sm100::f32x2 (&x)[4]) {
        const float2 a = sm100::unpack2(x[0]), b = sm100::unpack2(x[1]), c = sm100::unpack2(x[2]),
                     e = sm100::unpack2(x[3]);
        reinterpret_cast<float4 *>(p)[0] = make_float4(a.x, a.y, b.x, b.y);
        reinterpret_cast<float4 *>(p)[1] = make_float4(c.x, c.y, e.x, e.y);
    }
};

// One CTA per two consecutive runs of kRun tokens of one (tensor, head):
// both runs' TMA tiles are requested at the start, so the second one loads
// while the first is computed.  A group of D / 8 lanes owns a token (8
// channels per lane), so a warp works on 32 * 8 / D tokens at once; each
// group walks its own consecutive tokens with the three previous inputs in
// registers.  Six resident CTAs per SM keep twelve tiles in flight.
// PART 0 runs the q and k tensors (L2-normalised; beta with q), PART 1 the
// v tensor: the norm test is a compile-time constant in each instance.
template <typename Tin, int D, int PART>
__global__ void __launch_bounds__(kPrepWarps * 32, 6) prep_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                               PrepArgs a) {
    using namespace sm100;
    constexpr int CPL = 8;                       // channels per lane
    constexpr int LPT = D / CPL;                 // lanes per token
    constexpr int SLOTS = 32 / LPT;              // tokens per warp step
    constexpr int PER_WARP = kRun / kPrepWarps;
    constexpr int PER_SLOT = PER_WARP / SLOTS;   // consecutive tokens per lane group
    static_assert(PER_SLOT >= 1 && PER_WARP % SLOTS == 0, "run split");
    constexpr int TILE_BYTES = (kRun + kHalo) * D * static_cast<int>(sizeof(Tin));
    constexpr int TILE_STRIDE = prep_tile_bytes<Tin, D>();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *taps_t = reinterpret_cast<float *>(smem_raw + 2 * TILE_STRIDE);   // [4][D]: tap-major
    uint64_t *bars = reinterpret_cast<uint64_t *>(taps_t + 4 * D);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H;
    // task counts fit in 32 bits (the launcher checks): a CTA owns the runs
    // 2 rp, 2 rp + 1 of one (tensor, head) mh, or one empty sequence's state
    constexpr int M0 = PART == 0 ? 0 : 2, NM = PART == 0 ? 2 : 1;  // this instance's tensors
    const int row_tasks = NM * H;                                  // (tensor, head) pairs
    const int n_runs = (a.T_total + kRun - 1) / kRun;
    const int run_tasks = (n_runs + 1) / 2 * row_tasks;
    const int task = static_cast<int>(blockIdx.x);
    const Tin *sin = static_cast<const Tin *>(a.state_in);
    Tin *sout = static_cast<Tin *>(a.state_out);
    const size_t tok_x = static_cast<size_t>(3) * H * D;             // one token of x_qkv

    if (task >= run_tasks) {
        // conv state of an empty sequence passes through (or becomes zero)
        constexpr int CPE = D / 32;
        const int et = task - run_tasks;
        if (warp != 0 || et >= a.N * row_tasks || !sout) return;
        const int n = et / row_tasks;
        const int mh = M0 * H + et % row_tasks;
        int bos, eos;
        span_of(a, n, bos, eos);
        if (eos > bos) return;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const size_t o = (static_cast<size_t>(n) * 3 + j) * tok_x + static_cast<size_t>(mh) * D + lane * CPE;
            float w[CPE];
            if (sin) Lanes<Tin, CPE>::load(sin + o, w);
            else
#pragma unroll
                for (int i = 0; i < CPE; ++i) w[i] = 0.f;
            Lanes<Tin, CPE>::store(sout + o, w);
        }
        return;
    }

    const int run0 = task / row_tasks * 2;
    const int mh = M0 * H + task % row_tasks;              // m * H + h
    const int m = mh / H, h = mh % H;
    const int nr = min(2, n_runs - run0);                  // runs of this CTA
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)        // rows t_begin - 3 .. t_begin + 63 of each run of this (tensor, head); out of range -> 0
        for (int r = 0; r < nr; ++r) {
            mbar_arrive_expect_tx(&bars[r], TILE_BYTES);
            tma_load_3d(smem_raw + r * TILE_STRIDE, &tm_x, &bars[r], 0, mh, (run0 + r) * kRun - kHalo);
        }

    const int slot = lane / LPT, sl = lane % LPT;
    // conv taps of this lane's channels as (even, odd) pairs: wt[tap][pair], tap 3 = current token
    const int c0 = sl * CPL;
    // taps stored tap-major in shared memory, so one 16-byte load gives two (even, odd) channel pairs of
    // a tap; they are re-read per token rather than held in 32 registers
    if (tid < D) {
        const float4 w = __ldg(reinterpret_cast<const float4 *>(a.conv_w) + static_cast<size_t>(mh) * D + tid);
        taps_t[tid] = w.x; taps_t[D + tid] = w.y; taps_t[2 * D + tid] = w.z; taps_t[3 * D + tid] = w.w;
    }
    __syncthreads();
    auto load_taps = [&](f32x2 (&wt)[4][4]) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint64_t lo, hi;
                asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(lo), "=l"(hi)
                             : "r"(smem_u32(taps_t + k * D + c0 + 4 * h2)));
                wt[k][2 * h2] = lo;
                wt[k][2 * h2 + 1] = hi;
            }
    };
    const size_t col = static_cast<size_t>(mh) * D + c0;            // this lane's channels in a token of x
    Tin *dst = static_cast<Tin *>(m == 0 ? a.q : (m == 1 ? a.k : a.v)) + static_cast<size_t>(h) * D + c0;
    const size_t tok_o = static_cast<size_t>(H) * D;
#pragma unroll 1
    for (int r = 0; r < nr; ++r) {
        const Tin *tile = reinterpret_cast<const Tin *>(smem_raw + r * TILE_STRIDE);
        uint64_t *bar = &bars[r];
        const int t_begin = (run0 + r) * kRun, t_end = min(t_begin + kRun, a.T_total);
        const int s_begin = t_begin + warp * PER_WARP + slot * PER_SLOT;
        const int s_end = min(s_begin + PER_SLOT, t_end);
        int n = 0, bos = 0, eos = 0;
        if (s_begin < s_end) {
            n = seq_of(a, s_begin);
            span_of(a, n, bos, eos);
            while (eos <= s_begin && n + 1 < a.N) {      // empty sequences at s_begin
                ++n;
                span_of(a, n, bos, eos);
            }
        }
        // warp-uniform: every lane of a warp takes part in the group reductions below
        if (!__all_sync(0xffffffffu, mbar_wait(bar, 0, kPrepWaitNs))) {
            if (lane == 0) atomicAdd(&g_prep_timeouts, 1u);
            // this and the next run's tile copies may still be in flight into
            // this CTA's shared memory: one more bounded wait each before it exits
            for (int r2 = r; r2 < nr; ++r2) mbar_wait(&bars[r2], 0, kPrepWaitNs);
            return;
        }
        auto row_ptr = [&](int t) { return tile + static_cast<size_t>(t - t_begin + kHalo) * D + c0; };

        // window: x of the three tokens before the current one (win[0] oldest)
        f32x2 win[3][4] = {};
        auto fill_window = [&](int t) {              // window for token t of sequence n (bos <= t)
    #pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int p = t - 3 + j;
                if (p >= bos) {
                    Oct<Tin>::ld_shared(row_ptr(p), win[j]);
                } else if (sin) {
                    const int tap = p - bos + 3;     // 0..2: state token bos - 3 + tap
                    Oct<Tin>::ld_global(sin + (static_cast<size_t>(n) * 3 + tap) * tok_x + col, win[j]);
                } else {
    #pragma unroll
                    for (int q = 0; q < 4; ++q) win[j][q] = 0ull;
                }
            }
        };
        if (s_begin < s_end) fill_window(s_begin);
        const f32x2 nl2e = pack2(-1.4426950408889634f, -1.4426950408889634f), one = pack2(1.f, 1.f);
        // one token; Boundary: the run may cross a sequence end (else straight-line code)
        auto token = [&](int t, bool act, auto boundary) {
            if (decltype(boundary)::value && act && t >= eos) {                    // next sequence: restart the window
                do {
                    ++n;
                    span_of(a, n, bos, eos);
                } while (eos <= t && n + 1 < a.N);
                fill_window(t);
            }
            f32x2 wt[4][4];
            load_taps(wt);
            f32x2 xt[4], y[4], ss2 = 0ull;
            if (act) Oct<Tin>::ld_shared(row_ptr(t), xt);
            else
    #pragma unroll
                for (int q = 0; q < 4; ++q) xt[q] = 0ull;
    #pragma unroll
            for (int q = 0; q < 4; ++q) {
                f32x2 c = fmul2(wt[0][q], win[0][q]);
                c = ffma2(wt[1][q], win[1][q], c);
                c = ffma2(wt[2][q], win[2][q], c);
                c = ffma2(wt[3][q], xt[q], c);
                // Swish(c) = c / (1 + e^{-c})
                const float2 e = unpack2(fmul2(c, nl2e));
                float ex, ey;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ex) : "f"(e.x));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ey) : "f"(e.y));
                const float2 den = unpack2(fadd2(pack2(ex, ey), one));
                y[q] = fmul2(c, pack2(__fdividef(1.0f, den.x), __fdividef(1.0f, den.y)));
                ss2 = ffma2(y[q], y[q], ss2);
                win[0][q] = win[1][q];
                win[1][q] = win[2][q];
                win[2][q] = xt[q];
            }
            if constexpr (PART == 0) {                // q, k: L2Norm over the head's d channels
                const float2 s2 = unpack2(ss2);
                float ss = s2.x + s2.y;
    #pragma unroll
                for (int o = LPT / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float r = rsqrtf(ss + a.l2_eps);
                const f32x2 r2 = pack2(r, r);
    #pragma unroll
                for (int q = 0; q < 4; ++q) y[q] = fmul2(y[q], r2);
            }
            if (act) {
                Oct<Tin>::st_global(dst + static_cast<size_t>(t) * tok_o, y);
                if (decltype(boundary)::value && t == eos - 1 && sout) {           // last token: save the window as conv state
    #pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        Tin *sp = sout + (static_cast<size_t>(n) * 3 + j) * tok_x + col;
                        Oct<Tin>::st_global(sp, win[j]);
                    }
                }
            }
        };
        // fast path: every group's tokens are PER_SLOT tokens of one sequence
        const bool inside = s_end - s_begin == PER_SLOT && eos >= s_end;
        if (__all_sync(0xffffffffu, inside)) {
        #pragma unroll
            for (int u2 = 0; u2 < PER_SLOT; ++u2) token(s_begin + u2, true, std::false_type{});
            if (eos == s_end && sout) {           // the group ends its sequence: save the window
        #pragma unroll
                for (int j = 0; j < 3; ++j)
                    Oct<Tin>::st_global(sout + (static_cast<size_t>(n) * 3 + j) * tok_x + col, win[j]);
            }
        } else {
            for (int u2 = 0; u2 < PER_SLOT; ++u2) token(s_begin + u2, s_begin + u2 < s_end, std::true_type{});
        }
        // beta = Sigmoid(logit) for this run's tokens and head h (the q-tensor CTAs)
        if (PART == 0 && m == 0 && a.beta_logit) {
            const Tin *bl = static_cast<const Tin *>(a.beta_logit);
            Tin *bo = static_cast<Tin *>(a.beta);
            for (int t = t_begin + tid; t < t_end; t += kPrepWarps * 32)
                st_out(bo + static_cast<size_t>(t) * H + h, sigmoid(ld_in(bl + static_cast<size_t>(t) * H + h)));
        }

    }
}

template <typename Tin, int D>
__global__ void __launch_bounds__(kWarps * 32) output_gate_kernel(PostArgs a) {
    constexpr int CPL = D / 32;
    // bf16 rows are held as the loaded words and widened only when used, so
    // every row's loads are issued before the first one is waited on
    constexpr bool RAW = sizeof(Tin) == 2 && CPL == 4;
    constexpr int RPW = 4;                               // rows per warp
    const int lane = threadIdx.x & 31;
    const long long row0 = (static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * RPW;
    const Tin *o = static_cast<const Tin *>(a.o);
    const Tin *g = static_cast<const Tin *>(a.gate);
    Tin *y = static_cast<Tin *>(a.y);
    float w[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) w[i] = a.norm_w ? __ldg(a.norm_w + lane * CPL + i) : 1.f;
    if constexpr (RAW) {
        uint2 ow[RPW], gw[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            if (row0 + r >= a.rows) break;
            const size_t off = static_cast<size_t>(row0 + r) * D + lane * CPL;
            ow[r] = __ldg(reinterpret_cast<const uint2 *>(o + off));
            gw[r] = __ldg(reinterpret_cast<const uint2 *>(g + off));
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            if (row0 + r >= a.rows) break;
            const float ov[4] = {__uint_as_float(ow[r].x << 16), __uint_as_float(ow[r].x & 0xffff0000u),
                                  __uint_as_float(ow[r].y << 16), __uint_as_float(ow[r].y & 0xffff0000u)};
            const float gv[4] = {__uint_as_float(gw[r].x << 16), __uint_as_float(gw[r].x & 0xffff0000u),
                                  __uint_as_float(gw[r].y << 16), __uint_as_float(gw[r].y & 0xffff0000u)};
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) ss += ov[i] * ov[i];
            const float inv = rsqrtf(warp_sum(ss) / D + a.eps);
            float out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) out[i] = sigmoid(gv[i]) * (ov[i] * inv * w[i]);
            Lanes<Tin, CPL>::store(y + static_cast<size_t>(row0 + r) * D + lane * CPL, out);
        }
    } else {
        float ov[RPW][CPL], gv[RPW][CPL];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            if (row0 + r >= a.rows) break;
            const size_t off = static_cast<size_t>(row0 + r) * D + lane * CPL;
            Lanes<Tin, CPL>::load(o + off, ov[r]);
            Lanes<Tin, CPL>::load(g + off, gv[r]);
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            if (row0 + r >= a.rows) break;
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) ss += ov[r][i] * ov[r][i];
            const float inv = rsqrtf(warp_sum(ss) / D + a.eps);
            float out[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) out[i] = sigmoid(gv[r][i]) * (ov[r][i] * inv * w[i]);
            Lanes<Tin, CPL>::store(y + static_cast<size_t>(row0 + r) * D + lane * CPL, out);
        }
    }
}

// x_qkv [T, 3, H, d] viewed as the 3-D tensor (channel, tensor-head, token).
template <typename Tin, int D>
cudaError_t launch_prep_d(const PrepArgs &a, cudaStream_t s) {
    // per instance, a CTA per pair of runs of each of its (tensor, head)
    // pairs, then one per empty-sequence state: q and k (2 H pairs), v (H)
    const long long per_h = static_cast<long long>(((a.T_total + kRun - 1) / kRun + 1) / 2) +
                            static_cast<long long>(a.N);
    const long long tasks_qk = per_h * 2 * a.H, tasks_v = per_h * a.H;
    if (tasks_v <= 0) return cudaSuccess;
    if (tasks_qk > 0x7fffffffLL) return cudaErrorInvalidValue;
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorInvalidValue;
    CUtensorMap tm;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(3) * a.H,
                                static_cast<cuuint64_t>(a.T_total > 0 ? a.T_total : 1)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * sizeof(Tin),
                                   static_cast<cuuint64_t>(3) * a.H * D * sizeof(Tin)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(kRun + kHalo)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(&tm, sizeof(Tin) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                           3, const_cast<void *>(a.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    constexpr int smem = prep_smem_bytes<Tin, D>();
    if (smem > 48 * 1024) {
        cudaError_t ea = cudaFuncSetAttribute(prep_kernel<Tin, D, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (ea == cudaSuccess)
            ea = cudaFuncSetAttribute(prep_kernel<Tin, D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (ea != cudaSuccess) return ea;
    }
    prep_kernel<Tin, D, 0><<<static_cast<unsigned>(tasks_qk), kPrepWarps * 32, smem, s>>>(tm, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    prep_kernel<Tin, D, 1><<<static_cast<unsigned>(tasks_v), kPrepWarps * 32, smem, s>>>(tm, a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

template <typename Tin>
cudaError_t launch_prep_t(int d, const PrepArgs &a, cudaStream_t s) {
    if (d == 128) return launch_prep_d<Tin, 128>(a, s);
    if (d == 64) return launch_prep_d<Tin, 64>(a, s);
    if (d == 32) return launch_prep_d<Tin, 32>(a, s);
    return cudaErrorInvalidValue;
}

template <typename Tin>
cudaError_t launch_post_t(int d, const PostArgs &a, cudaStream_t s) {
    constexpr int rpw = 4;                       // the kernel's rows per warp
    const long long blocks = (a.rows + kWarps * rpw - 1) / (kWarps * rpw);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (d == 128) output_gate_kernel<Tin, 128><<<grid, kWarps * 32, 0, s>>>(a);
    else if (d == 64) output_gate_kernel<Tin, 64><<<grid, kWarps * 32, 0, s>>>(a);
    else if (d == 32) output_gate_kernel<Tin, 32><<<grid, kWarps * 32, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_prep(kda_dtype dt, int d, const PrepArgs &a, cudaStream_t s) {
    if (dt == KDA_BF16) return launch_prep_t<__nv_bfloat16>(d, a, s);
    return launch_prep_t<float>(d, a, s);
}

cudaError_t launch_output_gate(kda_dtype dt, int d, const PostArgs &a, cudaStream_t s) {
    if (dt == KDA_BF16) return launch_post_t<__nv_bfloat16>(d, a, s);
    return launch_post_t<float>(d, a, s);
}

unsigned int take_prep_timeouts() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_prep_timeouts, sizeof(v)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_prep_timeouts, &zero, sizeof(zero));
    return v;
}

}  // namespace kda
