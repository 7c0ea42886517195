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
// Both passes are HBM-bound streams.  prep: one CTA owns a run of 64
// consecutive tokens of one (tensor, head): one TMA copy brings the run and
// the three tokens before it ([67, d], rows before the first token read as
// zero) into shared memory, so many runs are in flight per SM without
// holding registers; each of four warps then walks 16 tokens with the
// three previous inputs of its lane's d/32 channels in registers, the L2
// norm as a warp reduction.  Inputs before a sequence's first token come
// from the caller's conv state (or zero), never from the previous sequence.
// post: one warp per (token, head) row, four rows per warp in flight.
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
template <typename T, int CPL>
__device__ __forceinline__ void load_row(const T *p, float (&x)[CPL]) {
    if constexpr (CPL == 4 && sizeof(T) == 2) {
        const uint2 w = *reinterpret_cast<const uint2 *>(p);
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&w.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w.y);
        x[0] = __low2float(a); x[1] = __high2float(a); x[2] = __low2float(b); x[3] = __high2float(b);
    } else if constexpr (CPL == 4) {
        const float4 w = *reinterpret_cast<const float4 *>(p);
        x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
    } else {
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            if constexpr (sizeof(T) == 2) x[i] = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
            else x[i] = reinterpret_cast<const float *>(p)[i];
        }
    }
}

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
__device__ __forceinline__ float swish(float x) { return x * sigmoid(x); }

// Swish of a channel pair: the exponentials and reciprocals stay per lane
// (MUFU), the rest is packed.  Same arithmetic as swish() per element.
__device__ __forceinline__ sm100::f32x2 swish2(sm100::f32x2 c) {
    using namespace sm100;
    const float2 m = unpack2(fmul2(c, pack2(-1.4426950408889634f, -1.4426950408889634f)));
    float ex, ey;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ex) : "f"(m.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ey) : "f"(m.y));
    const float2 den = unpack2(fadd2(pack2(ex, ey), pack2(1.f, 1.f)));
    return fmul2(c, pack2(__fdividef(1.0f, den.x), __fdividef(1.0f, den.y)));
}

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
constexpr int prep_smem_bytes() {
    return (((kRun + kHalo) * D * static_cast<int>(sizeof(Tin)) + 15) & ~15) + 16;   // tile + mbarrier
}

template <typename Tin, int D>
__global__ void __launch_bounds__(kPrepWarps * 32) prep_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                               PrepArgs a) {
    using namespace sm100;
    constexpr int CPL = D / 32;                 // channels per lane
    constexpr int TILE_BYTES = (kRun + kHalo) * D * static_cast<int>(sizeof(Tin));
    constexpr int PER_WARP = kRun / kPrepWarps;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const Tin *tile = reinterpret_cast<const Tin *>(smem_raw);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw + ((TILE_BYTES + 15) & ~15));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H;
    const long long row_tasks = static_cast<long long>(3) * H;     // (tensor, head) pairs
    const long long run_tasks = static_cast<long long>((a.T_total + kRun - 1) / kRun) * row_tasks;
    const long long task = blockIdx.x;
    const Tin *x = static_cast<const Tin *>(a.x);
    const Tin *sin = static_cast<const Tin *>(a.state_in);
    Tin *sout = static_cast<Tin *>(a.state_out);
    const size_t tok_x = static_cast<size_t>(3) * H * D;             // one token of x_qkv

    if (task >= run_tasks) {
        // conv state of an empty sequence passes through (or becomes zero)
        const long long et = task - run_tasks;
        if (warp != 0 || et >= static_cast<long long>(a.N) * row_tasks || !sout) return;
        const int n = static_cast<int>(et / row_tasks);
        const int mh = static_cast<int>(et % row_tasks);
        int bos, eos;
        span_of(a, n, bos, eos);
        if (eos > bos) return;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const size_t o = (static_cast<size_t>(n) * 3 + j) * tok_x + static_cast<size_t>(mh) * D + lane * CPL;
            float w[CPL];
            if (sin) Lanes<Tin, CPL>::load(sin + o, w);
            else
#pragma unroll
                for (int i = 0; i < CPL; ++i) w[i] = 0.f;
            Lanes<Tin, CPL>::store(sout + o, w);
        }
        return;
    }

    const int run = static_cast<int>(task / row_tasks);
    const int mh = static_cast<int>(task % row_tasks);     // m * H + h
    const int m = mh / H, h = mh % H;
    const int t_begin = run * kRun, t_end = min(t_begin + kRun, a.T_total);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {      // rows t_begin - 3 .. t_begin + 63 of this (tensor, head); out of range -> 0
        mbar_arrive_expect_tx(bar, TILE_BYTES);
        tma_load_3d(smem_raw, &tm_x, bar, 0, mh, t_begin - kHalo);
    }

    // conv taps of this lane's channels: w[ch][0..3], tap 3 = current token
    const size_t col = static_cast<size_t>(mh) * D + lane * CPL;   // this lane's channels in a token of x
    float wt[CPL][4];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        const float4 w4 = __ldg(reinterpret_cast<const float4 *>(a.conv_w) + static_cast<size_t>(mh) * D + lane * CPL + i);
        wt[i][0] = w4.x; wt[i][1] = w4.y; wt[i][2] = w4.z; wt[i][3] = w4.w;
    }
    Tin *dst = static_cast<Tin *>(m == 0 ? a.q : (m == 1 ? a.k : a.v));
    const size_t tok_o = static_cast<size_t>(H) * D;
    const int w_begin = t_begin + warp * PER_WARP, w_end = min(w_begin + PER_WARP, t_end);
    int n = 0, bos = 0, eos = 0;
    if (w_begin < w_end) {
        n = seq_of(a, w_begin);
        span_of(a, n, bos, eos);
        while (eos <= w_begin && n + 1 < a.N) {      // empty sequences at w_begin
            ++n;
            span_of(a, n, bos, eos);
        }
    }
    if (!mbar_wait(bar, 0, kPrepWaitNs)) {
        if (lane == 0) atomicAdd(&g_prep_timeouts, 1u);
        return;
    }
    auto row_ptr = [&](int t) { return tile + static_cast<size_t>(t - t_begin + kHalo) * D + lane * CPL; };

    // window: x of the three tokens before the current one (win[0] oldest)
    float win[3][CPL];
    auto fill_window = [&](int t) {              // window for token t of sequence n (bos <= t)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int p = t - 3 + j;
            if (p >= bos) {
                load_row<Tin, CPL>(row_ptr(p), win[j]);
            } else if (sin) {
                const int tap = p - bos + 3;     // 0..2: state token bos - 3 + tap
                Lanes<Tin, CPL>::load(sin + (static_cast<size_t>(n) * 3 + tap) * tok_x + col, win[j]);
            } else {
#pragma unroll
                for (int i = 0; i < CPL; ++i) win[j][i] = 0.f;
            }
        }
    };
    if (w_begin < w_end) fill_window(w_begin);
#pragma unroll 2
    for (int t = w_begin; t < w_end; ++t) {
        if (t >= eos) {                           // next sequence: restart the window
            do {
                ++n;
                span_of(a, n, bos, eos);
            } while (eos <= t && n + 1 < a.N);
            fill_window(t);
        }
        float xt[CPL];
        load_row<Tin, CPL>(row_ptr(t), xt);
        float y[CPL];
        float ss = 0.f;
        if constexpr (CPL == 4) {                 // channel pairs in f32x2
            using namespace sm100;
            f32x2 ss2 = 0ull;
#pragma unroll
            for (int p2 = 0; p2 < 2; ++p2) {
                const int i0 = 2 * p2, i1 = i0 + 1;
                const f32x2 x2 = pack2(xt[i0], xt[i1]);
                f32x2 c = fmul2(pack2(wt[i0][0], wt[i1][0]), pack2(win[0][i0], win[0][i1]));
                c = ffma2(pack2(wt[i0][1], wt[i1][1]), pack2(win[1][i0], win[1][i1]), c);
                c = ffma2(pack2(wt[i0][2], wt[i1][2]), pack2(win[2][i0], win[2][i1]), c);
                c = ffma2(pack2(wt[i0][3], wt[i1][3]), x2, c);
                const f32x2 yy = swish2(c);
                ss2 = ffma2(yy, yy, ss2);
                const float2 yv = unpack2(yy);
                y[i0] = yv.x;
                y[i1] = yv.y;
            }
            const float2 s2 = unpack2(ss2);
            ss = s2.x + s2.y;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                win[0][i] = win[1][i];
                win[1][i] = win[2][i];
                win[2][i] = xt[i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const float c = wt[i][0] * win[0][i] + wt[i][1] * win[1][i] + wt[i][2] * win[2][i] + wt[i][3] * xt[i];
                y[i] = swish(c);
                ss += y[i] * y[i];
                win[0][i] = win[1][i];
                win[1][i] = win[2][i];
                win[2][i] = xt[i];
            }
        }
        if (m < 2) {                              // q, k: L2Norm over the head's d channels
            const float r = rsqrtf(warp_sum(ss) + a.l2_eps);
#pragma unroll
            for (int i = 0; i < CPL; ++i) y[i] *= r;
        }
        Lanes<Tin, CPL>::store(dst + static_cast<size_t>(t) * tok_o + static_cast<size_t>(h) * D + lane * CPL, y);
        if (t == eos - 1 && sout) {               // last token: save the window as conv state
#pragma unroll
            for (int j = 0; j < 3; ++j)
                Lanes<Tin, CPL>::store(sout + (static_cast<size_t>(n) * 3 + j) * tok_x + col, win[j]);
        }
    }
    // beta = Sigmoid(logit) for this run's tokens and head h (the q-tensor CTAs)
    if (m == 0 && a.beta_logit) {
        const Tin *bl = static_cast<const Tin *>(a.beta_logit);
        Tin *bo = static_cast<Tin *>(a.beta);
        for (int t = t_begin + tid; t < t_end; t += kPrepWarps * 32)
            st_out(bo + static_cast<size_t>(t) * H + h, sigmoid(ld_in(bl + static_cast<size_t>(t) * H + h)));
    }
}

template <typename Tin, int D>
__global__ void __launch_bounds__(kWarps * 32) output_gate_kernel(PostArgs a) {
    constexpr int CPL = D / 32;
    constexpr int RPW = 4;                       // rows per warp
    const int lane = threadIdx.x & 31;
    const long long row0 = (static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * RPW;
    const Tin *o = static_cast<const Tin *>(a.o);
    const Tin *g = static_cast<const Tin *>(a.gate);
    Tin *y = static_cast<Tin *>(a.y);
    float w[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) w[i] = a.norm_w ? __ldg(a.norm_w + lane * CPL + i) : 1.f;
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

// x_qkv [T, 3, H, d] viewed as the 3-D tensor (channel, tensor-head, token).
template <typename Tin, int D>
cudaError_t launch_prep_d(const PrepArgs &a, cudaStream_t s) {
    const long long tasks = static_cast<long long>((a.T_total + kRun - 1) / kRun) * 3 * a.H +
                            static_cast<long long>(a.N) * 3 * a.H;
    if (tasks <= 0) return cudaSuccess;
    if (tasks > 0x7fffffffLL) return cudaErrorInvalidValue;
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
    prep_kernel<Tin, D><<<static_cast<unsigned>(tasks), kPrepWarps * 32, smem, s>>>(tm, a);
    const cudaError_t e = cudaGetLastError();
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
    const long long blocks = (a.rows + kWarps * 4 - 1) / (kWarps * 4);
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
