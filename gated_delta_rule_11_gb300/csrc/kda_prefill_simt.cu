// Chunked KDA prefill on the CUDA cores (fp32 FFMA throughout).
//
// This kernel serves the fp32 path (whose tolerance the tensor cores' bf16
// and tf32 operands cannot meet) and every head-dimension combination.  One
// CTA owns one (sequence, head) chain and one dv/4-column slab of the value
// dimension: the value columns of the state never interact, so slabs are
// independent (the key-side work of a tile is recomputed per slab), and
// four CTAs per chain keep several chains' latency-bound tiles in flight
// per SM at every head size.
//
// Per 16-token tile (the tile of "Kimi K3：从三条信息流到完整系统",
// §下界 log-decay 是一个 kernel 设计, whose bound -80 < sum g < 0 keeps
// e^{-b} finite in fp32), with b_r the inclusive in-tile cumulative sum of
// the eq. (5) log-decay and S_0 the state entering the tile:
//   L  = StrictTril[(K*e^b)(K*e^-b)^T]       A = Tril[(Q*e^b)(K*e^-b)^T]
//   (I + Diag(beta) L) [U | W] = Diag(beta) [V | K*e^b]   (forward substitution)
//   Vt = U - W S_0
//   O  = scale * ((Q*e^b) S_0 + A Vt)
//   S  = Diag(e^{b_C}) S_0 + (K*e^{b_C - b})^T Vt
// which is eq. (4) of §从投影到 Chunkwise 的完整接口 with the UT transform
// written out (Tril keeps the diagonal: a token reads its own write).
// Tokens past the end of a sequence enter the last tile as k = q = v = 0,
// beta = 0, g = 0, which leaves the state untouched.
//
// Gate variants (kda_gate_mode): the log-decay g comes from the gate input
// under the chosen map, per key channel or one per head.  An unbounded gate
// (the log-decay itself, or Kimi Linear's negative softplus, "Kimi K3: Two
// point eight trillion parameters, open weights, and forty-seven pages of
// how", §What changed between the paper and the model) can drive b far
// below -80 within a tile, where e^{-b} overflows; for those the kernel
// takes the position-pair path that the bound was introduced to avoid:
//   L_rs = sum_c k_rc k_sc e^{b_rc - b_sc},  A_rs = sum_c q_rc k_sc e^{b_rc - b_sc}
// (s <= r, so every exponent is <= 0), with the other factors unchanged
// (e^{b}, e^{b_C - b} <= 1 never overflow).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = 16;      // tile length (tokens)
constexpr int NT = 128;    // threads per CTA

template <int DK, int BV>
struct SimtSmem {
    float kg[C][DK], kinv[C][DK], qg[C][DK], kdec[C][DK], W[C][DK];
    float S[DK][BV];
    float vv[C][BV], U[C][BV], Vt[C][BV];
    float L[C][C], A[C][C];
    float beta[C];
    float ebC[DK];
};
// Extra shared memory of the position-pair path: raw k, raw q (masked) and b.
template <int DK>
struct SimtPairSmem {
    float k[C][DK], q[C][DK], b[C][DK];
};

// BV value columns per CTA (a quarter of dv, so every head size has four
// slabs per chain); value-side thread (j, rg): column j = tid % BV of row
// group rg = tid / BV, tile rows rg + m * RG.
template <typename Tin, int DK, int DV, int BV>
__global__ void __launch_bounds__(NT) prefill_simt_kernel(PrefillArgs a) {
    constexpr int RG = NT / BV;        // row groups
    constexpr int RPT = C / RG;        // tile rows per thread in the value-side products
    static_assert(NT % BV == 0 && C % RG == 0 && DK % RG == 0, "value-side tiling");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem<DK, BV> &sm = *reinterpret_cast<SimtSmem<DK, BV> *>(smem_raw);
    SimtPairSmem<DK> &pp = *reinterpret_cast<SimtPairSmem<DK> *>(smem_raw + sizeof(SimtSmem<DK, BV>));
    const bool pairs = a.gate_mode == KDA_GATE_LOG_DECAY || a.gate_mode == KDA_GATE_NEG_SOFTPLUS;

    const int tid = threadIdx.x, lane = tid & 31;
    const int chain = blockIdx.x;             // n * H + h
    const int n = chain / a.H, h = chain % a.H;
    const int j0 = blockIdx.y * BV;
    int bos, eos;
    seq_span(a, n, bos, eos);
    const float escale = a.A_log ? expf(__ldg(a.A_log + h)) : 1.0f;

    const Tin *gq = static_cast<const Tin *>(a.q);
    const Tin *gk = static_cast<const Tin *>(a.k);
    const Tin *gv = static_cast<const Tin *>(a.v);
    const Tin *gz = static_cast<const Tin *>(a.g);
    const Tin *gb = static_cast<const Tin *>(a.beta);
    Tin *go = static_cast<Tin *>(a.out);
    const size_t tok_k = static_cast<size_t>(a.H) * DK, tok_v = static_cast<size_t>(a.H) * DV;
    const size_t state_off = static_cast<size_t>(chain) * DK * DV;

    for (int idx = tid; idx < DK * BV; idx += NT) {
        const int c = idx / BV, j = idx % BV;
        sm.S[c][j] = a.init_state ? a.init_state[state_off + static_cast<size_t>(c) * DV + j0 + j] : 0.f;
    }

    const long long ck_row0 = a.ckpt ? ckpt_first_row(a, n) : 0;
    for (int t0 = bos; t0 < eos; t0 += C) {
        const int nv = min(C, eos - t0);
        __syncthreads();  // previous tile is done with shared memory

        // Gate, in-tile cumulative log-decay and the decay-scaled operands.
        // All of the tile's loads are issued before any is used (rows past
        // the sequence end re-read its last row and are masked below).
        for (int c = tid; c < DK; c += NT) {
            float zr[C], kr[C], qr[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const size_t tok = static_cast<size_t>(t0 + min(r, nv - 1));
                const size_t off = tok * tok_k + h * DK + c;
                zr[r] = a.gate_mode == KDA_GATE_NONE
                            ? 0.f : ld_in(gz + (a.gate_scalar ? tok * a.H + h : off));
                kr[r] = ld_in(gk + off);
                qr[r] = ld_in(gq + off);
            }
            float b[C];
            float run = 0.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                if (r < nv) run += gate_log_decay(a.gate_mode, zr[r], escale, a.g_min);
                else kr[r] = qr[r] = 0.f;
                b[r] = run;
            }
            const float bC = run;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const float eb = expf(b[r]);
                sm.kg[r][c] = kr[r] * eb;
                sm.qg[r][c] = qr[r] * eb;
                sm.kdec[r][c] = kr[r] * expf(bC - b[r]);
                if (pairs) {
                    pp.k[r][c] = kr[r];
                    pp.q[r][c] = qr[r];
                    pp.b[r][c] = b[r];
                } else {
                    sm.kinv[r][c] = kr[r] * expf(-b[r]);
                }
            }
            sm.ebC[c] = expf(bC);
        }
        for (int idx = tid; idx < C * BV; idx += NT) {
            const int r = idx / BV, j = idx % BV;
            const float x = ld_in(gv + static_cast<size_t>(t0 + min(r, nv - 1)) * tok_v + h * DV + j0 + j);
            sm.vv[r][j] = r < nv ? x : 0.f;
        }
        if (tid < C) sm.beta[tid] = tid < nv ? ld_in(gb + static_cast<size_t>(t0 + tid) * a.H + h) : 0.f;
        __syncthreads();

        // L (strictly lower) and A (lower, diagonal kept): one entry (r, i)
        // per thread and pass, the whole dot product over c in-thread (no
        // shuffle chains on the critical path); each lane starts at its own
        // channel, so the 32 lanes' row reads hit 32 different banks.
#pragma unroll
        for (int pass = 0; pass < (C * C) / NT; ++pass) {
            const int e = tid + pass * NT;
            const int r = e / C, i = e % C;
            float l0 = 0.f, l1 = 0.f, a0 = 0.f, a1 = 0.f;
            if (i <= r) {
                if (pairs) {
#pragma unroll 4
                    for (int j = 0; j < DK; j += 2) {
                        const int c0 = (lane + j) & (DK - 1), c1 = (lane + j + 1) & (DK - 1);
                        const float k0 = pp.k[i][c0] * expf(pp.b[r][c0] - pp.b[i][c0]);
                        const float k1 = pp.k[i][c1] * expf(pp.b[r][c1] - pp.b[i][c1]);
                        l0 = fmaf(pp.k[r][c0], k0, l0);
                        a0 = fmaf(pp.q[r][c0], k0, a0);
                        l1 = fmaf(pp.k[r][c1], k1, l1);
                        a1 = fmaf(pp.q[r][c1], k1, a1);
                    }
                } else {
#pragma unroll 4
                    for (int j = 0; j < DK; j += 2) {
                        const int c0 = (lane + j) & (DK - 1), c1 = (lane + j + 1) & (DK - 1);
                        const float k0 = sm.kinv[i][c0], k1 = sm.kinv[i][c1];
                        l0 = fmaf(sm.kg[r][c0], k0, l0);
                        a0 = fmaf(sm.qg[r][c0], k0, a0);
                        l1 = fmaf(sm.kg[r][c1], k1, l1);
                        a1 = fmaf(sm.qg[r][c1], k1, a1);
                    }
                }
            }
            sm.L[r][i] = i < r ? l0 + l1 : 0.f;
            sm.A[r][i] = i <= r ? a0 + a1 : 0.f;
        }
        __syncthreads();

        // Forward substitution (the UT transform): one column per thread.
        for (int c = tid; c < DK; c += NT) {
            float w[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float acc = sm.kg[r][c];
#pragma unroll
                for (int i = 0; i < r; ++i) acc -= sm.L[r][i] * w[i];
                w[r] = sm.beta[r] * acc;
                sm.W[r][c] = w[r];
            }
        }
        for (int j = tid; j < BV; j += NT) {
            float u[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float acc = sm.vv[r][j];
#pragma unroll
                for (int i = 0; i < r; ++i) acc -= sm.L[r][i] * u[i];
                u[r] = sm.beta[r] * acc;
                sm.U[r][j] = u[r];
            }
        }
        __syncthreads();

        // Vt = U - W S_0 and the inter-tile output (Q*e^b) S_0.
        const int j = tid % BV, rg = tid / BV;
        float accw[RPT], accq[RPT];
#pragma unroll
        for (int m = 0; m < RPT; ++m) accw[m] = accq[m] = 0.f;
        for (int c = 0; c < DK; ++c) {
            const float s = sm.S[c][j];
#pragma unroll
            for (int m = 0; m < RPT; ++m) {
                const int r = rg + m * RG;
                accw[m] += sm.W[r][c] * s;
                accq[m] += sm.qg[r][c] * s;
            }
        }
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int r = rg + m * RG;
            sm.Vt[r][j] = sm.U[r][j] - accw[m];
        }
        __syncthreads();

        // Intra-tile output and the state update.
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int r = rg + m * RG;
            float o = accq[m];
            for (int i = 0; i <= r; ++i) o += sm.A[r][i] * sm.Vt[i][j];
            if (r < nv) st_out(go + (t0 + r) * tok_v + h * DV + j0 + j, a.scale * o);
        }
        float vt[C];
#pragma unroll
        for (int r = 0; r < C; ++r) vt[r] = sm.Vt[r][j];
        for (int c = rg; c < DK; c += RG) {
            float acc = sm.ebC[c] * sm.S[c][j];
#pragma unroll
            for (int r = 0; r < C; ++r) acc += sm.kdec[r][c] * vt[r];
            sm.S[c][j] = acc;
        }
        if (float *cp = ckpt_slot(a, ck_row0, t0 + nv - bos, h, static_cast<size_t>(DK) * DV)) {
            __syncthreads();   // uniform: every thread sees the same slot
            for (int idx = tid; idx < DK * BV; idx += NT) {
                const int c = idx / BV, jj = idx % BV;
                cp[static_cast<size_t>(c) * DV + j0 + jj] = sm.S[c][jj];
            }
        }
    }
    __syncthreads();
    if (a.final_state) {
        for (int idx = tid; idx < DK * BV; idx += NT) {
            const int c = idx / BV, jj = idx % BV;
            a.final_state[state_off + static_cast<size_t>(c) * DV + j0 + jj] = sm.S[c][jj];
        }
    }
}

template <typename Tin, int DK, int DV>
cudaError_t launch_one(const PrefillArgs &a, cudaStream_t s) {
    constexpr int BV = DV / 4;         // four value slabs per chain at every head size
    const bool pairs = a.gate_mode == KDA_GATE_LOG_DECAY || a.gate_mode == KDA_GATE_NEG_SOFTPLUS;
    const size_t smem = sizeof(SimtSmem<DK, BV>) + (pairs ? sizeof(SimtPairSmem<DK>) : 0);
    auto kern = prefill_simt_kernel<Tin, DK, DV, BV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sizeof(SimtSmem<DK, BV>) + sizeof(SimtPairSmem<DK>)));
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(a.N) * static_cast<unsigned>(a.H), DV / BV);
    kern<<<grid, NT, smem, s>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

template <typename Tin>
cudaError_t launch_t(int dk, int dv, const PrefillArgs &a, cudaStream_t s) {
#define KDA_SIMT_CASE(DK_, DV_) \
    if (dk == DK_ && dv == DV_) return launch_one<Tin, DK_, DV_>(a, s);
    KDA_SIMT_CASE(32, 32) KDA_SIMT_CASE(32, 64) KDA_SIMT_CASE(32, 128)
    KDA_SIMT_CASE(64, 32) KDA_SIMT_CASE(64, 64) KDA_SIMT_CASE(64, 128)
    KDA_SIMT_CASE(128, 32) KDA_SIMT_CASE(128, 64) KDA_SIMT_CASE(128, 128)
#undef KDA_SIMT_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_simt(kda_dtype dt, int dk, int dv, const PrefillArgs &a,
                                cudaStream_t s) {
    if (dt == KDA_BF16) return launch_t<__nv_bfloat16>(dk, dv, a, s);
    return launch_t<float>(dk, dv, a, s);
}

}  // namespace kda
