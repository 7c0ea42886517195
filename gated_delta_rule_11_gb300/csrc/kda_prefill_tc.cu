// Chunked KDA prefill on the 5th-generation tensor cores (tcgen05 + TMEM,
// TMA-fed): bf16 inputs, fp32 state, dk = dv = 128.
//
// Method ("Kimi K3：从三条信息流到完整系统"): the recurrence of §KDA 是带逐通道
// 遗忘的 delta rule, eq. (1), evaluated in the chunkwise form of
// §从投影到 Chunkwise 的完整接口, eqs. (3)-(4), over 16-token tiles -- the
// tile whose cumulative log-decay §下界 log-decay 是一个 kernel 设计 bounds to
// (-80, 0), so e^{-b} stays finite and the in-tile products are dense
// matmuls.  With b_r the in-tile inclusive cumsum of g, S_0 the state
// entering the tile, and the UT transform written out:
//   L  = StrictTril[(K e^b)(K e^-b)^T],   A = Tril[(Q e^b)(K e^-b)^T]
//   T  = (I + Diag(beta) L)^-1,  U = T Diag(beta) V,  W = T Diag(beta) (K e^b)
//   Vt = U - W S_0
//   O  = scale * ((Q e^b) S_0 + A Vt)
//   S  = Diag(e^{b_C}) S_0 + (K e^{b_C - b})^T Vt
//
// Precision.  Vt is the delta-rule residual (about |v|, while S is about
// 0.1-0.5), and rounding it, or A, to bf16 alone costs ~2e-2 of the output
// RMS.  So the tensor-core operands are fp16 (11-bit significand; every one
// of S, W, Q e^b, Vt, A, K e^{b_C-b} is bounded well inside fp16's range),
// L and A come from tf32 mma.sync on fp32 operands (K e^-b reaches e^80, out
// of fp16 range), and U, W, T, the gates and the state master are fp32.
// U is a bf16 product: v is bf16 already, and T Diag(beta) (tf32-rounded,
// 11 significant bits) is split exactly into bf16 hi + lo parts.
//
// Every tensor-core product is computed transposed so that its M side is a
// 128-wide head dimension (tcgen05 M = 128, TMEM lane j = value channel j):
// The chain writes the two operands it produces (the fp16 copy of S^T and
// Vt^T) straight into tensor memory, where the MMAs read them as A.  A
// tcgen05.mma occupies its issuing thread for ~110 cycles whatever its N
// (measured), while different threads' MMAs proceed concurrently; so (e) is
// split over 4 independent accumulators (K slices p, p + 4) issued by 4
// threads at once and summed by the chain, and (g), (h) are issued by two.
//   (e) E[:, 0:32]   = S^T [-W ; Q e^b]^T                M128 N32  K128
//       -> E[:, 0:16] = -(W S_0)^T, E[:, 16:32] = ((Q e^b) S_0)^T
//   (g) E[:, 16:32] += Vt^T A^T                          M128 N16  K16
//       -> E[:, 16:32] = O^T / scale
//   (h) H[:, 0:128]  = Vt^T (K e^{b_C - b})              M128 N128 K16
//       -> the state increment, transposed
//   (u) U^T = V^T (T Diag(beta))^T, hi + lo               M128 N16  K16 (x2)
//       -> read by the chain from TMEM (two slots, tile parity); V comes
//          from TMA in the 128B-swizzled MN-major operand layout
// E is double-buffered in TMEM (tile parity), so tile t's O is read out
// while tile t+1's (g)/(h) run, off the serial path; full tiles of O are
// staged in shared memory and written with one TMA store.
//
// CTA roles (one CTA per (sequence, head) chain, 512 threads):
//   warps 0-7  chain     : two warpgroups; thread (j, half) owns rows
//                          [64 half, 64 half + 64) of column j of the fp32
//                          state in registers.  Per tile they form
//                          Vt^T = U^T + D[:,0:16] as the fp16 operand of
//                          (g)/(h), store O, apply S = Diag(e^{b_C}) S +
//                          increment and write the fp16 copy of S^T (into
//                          TMEM) that the next tile's (e) reads.  Elected chain threads
//                          issue the tcgen05 products ((u) for the next tile by
//                          a thread idle while (e) runs) and commit them, and
//                          the TMA loads of the q, k, g_raw, v tiles (16
//                          tokens each) into a 4-stage ring, refilling a
//                          stage as soon as the chain has finished with it.
//   warps 8-15 producer  : two warpgroups taking alternate tiles, each with
//                          its own scratch; thread c owns key channel c: gate (eq. 5) and
//                          in-tile decays as running products of the
//                          retentions, decay-scaled operands, L and A (one
//                          16x8 block per warp), the triangular solve
//                          (first warp only, one barrier), W (tf32 mma.sync)
//                          and the bf16 hi/lo operand of (u).
// The chain is serial per tile; the producer and TMA run up to 3 tiles ahead.
// Tokens past a sequence's end are masked in the producer (k = q = 0, g = 0,
// beta = 0), which makes U, W, A and the increment vanish for them.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"
#include "kda_tc_util.cuh"

namespace kda {

__device__ unsigned int g_tc_timeouts = 0;

namespace {
using namespace sm100;
using namespace tcu;

constexpr int D = 128;           // dk = dv
constexpr int C = 16;            // tile tokens
constexpr int NS = 4;            // ring stages
constexpr int NTHREADS = 512;
constexpr int NPROD = 2;           // producer warpgroups
constexpr int NCHAIN = 256;        // chain threads (two warpgroups)
constexpr int TBS = 20;            // row stride of the fp32 T Diag(beta) tile (conflict-free fragments)
constexpr int TMEM_COLS = 512;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s (legitimate ones take microseconds)
constexpr int PADF = 132;        // fp32 row stride of the mma.sync operand tiles (conflict-free fragments)

// ---- shared memory map (bytes from a 1024-aligned base); stage s at s * STAGE_BYTES
constexpr int ST_Q = 0;          // [16][128] bf16 (TMA, unswizzled)
constexpr int ST_K = 4096;
constexpr int ST_Z = 8192;
constexpr int ST_V = 12288;      // A of U^T: bf16 MN-major SW128 (TMA, two 64-channel boxes)
constexpr int ST_WQ = 16384;     // B of (e): fp16 K-major SW128, 32 rows x 128 (rows 0-15 -W, 16-31 Q e^b)
constexpr int ST_KD = 24576;     // B of (h): fp16 MN-major SW128, mn = c, k = s
constexpr int ST_AT = 28672;     // B of (g): fp16 K-major none, 16 rows x 16
constexpr int ST_TB = 29696;     // B of U^T: bf16 K-major none, T Diag(beta) split hi | lo (16 x 16 each)
constexpr int ST_GC = 37888;     // fp32 [128] e^{b_C}
constexpr int ST_BETA = 38400;   // fp32 [16]
constexpr int STAGE_BYTES = 38912;
constexpr int OFF_OST = NS * STAGE_BYTES;         // two bf16 [16][128] O staging tiles (TMA store)
constexpr int OFF_VT = OFF_OST + 2 * C * D * 2;
constexpr int OFF_SCR = OFF_VT;                   // per-producer scratch, SCR_BYTES each:
constexpr int SC_KGM = 0;                         //   fp32 [16][PADF]: K e^b   (tf32-rounded)
constexpr int SC_QGM = C * PADF * 4;              //   fp32 [16][PADF]: Q e^b   (tf32-rounded)
constexpr int SC_KIM = 2 * C * PADF * 4;          //   fp32 [16][PADF]: K e^-b  (tf32-rounded)
constexpr int LSS = 20;                           //   row stride of L (16-byte aligned rows)
constexpr int SC_LS = 3 * C * PADF * 4;           //   fp32 [16][LSS]: L
constexpr int SC_TBF = SC_LS + C * LSS * 4;       //   fp32 [16][TBS]: T Diag(beta) (tf32-rounded)
constexpr int SC_T11 = SC_TBF + C * TBS * 4;      //   fp32 [8][8]: lower-right block of T (solve)
constexpr int SC_T00 = SC_T11 + 64 * 4;           //   fp32 [8][8]: upper-left block of T
constexpr int SC_Y = SC_T00 + 64 * 4;             //   fp32 [8][8]: Diag(beta) L10 T00
constexpr int SCR_BYTES = (SC_Y + 64 * 4 + 127) & ~127;
constexpr int OFF_BAR = (OFF_SCR + NPROD * SCR_BYTES + 63) & ~63;
enum { B_RAW = 0, B_FULL = NS, B_VT = 2 * NS, B_UPD, B_DRAIN, NUM_BARS };
constexpr int NACC = 4;          // independent accumulators of (e)
constexpr uint32_t TM_E = 0;     // two E buffers of NACC x 32 columns
constexpr uint32_t TM_H = 256;   // 128-column H
constexpr uint32_t TM_ST = 384;  // S^T fp16, 128 K values packed in 64 columns
constexpr uint32_t TM_VT = 448;  // Vt^T fp16, 16 K values packed in 8 columns
constexpr uint32_t TM_U = 464;   // two U^T slots of 16 columns (tile parity)
constexpr uint32_t E_BUF = NACC * 32;
constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_FLAG = OFF_SLOT + 4;
constexpr int SMEM_USED = OFF_FLAG + 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;      // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
static_assert(STAGE_BYTES % 1024 == 0 && ST_WQ % 1024 == 0 && ST_KD % 1024 == 0,
              "128B-swizzled operands need 1024-byte alignment");
constexpr uint32_t TX_BYTES = 4 * C * D * 2;        // q, k, g_raw, v tiles
constexpr uint32_t TX_BYTES_NOZ = 3 * C * D * 2;    // q, k, v (gate per head or none)

// The kernel's gate map (a compile-time instance parameter): the bounded
// map of eq. (5), or an unbounded one (the gate is the log-decay itself, or
// Kimi Linear's negative softplus).
enum : int { MAP_BOUNDED = 0, MAP_LOG_DECAY = 1, MAP_NEG_SOFTPLUS = 2 };
// The gate's shape (an instance parameter): decided at run time, or one
// input per key channel, or one per (token, head).
enum : int { SHAPE_ANY = 0, SHAPE_CHANNEL = 1, SHAPE_HEAD = 2 };
// log2 of the retention under an unbounded gate map: the gate itself, or
// -softplus(e^A z) = -(max(x, 0) + log(1 + e^-|x|)), in log2 units.
template <int Map>
__device__ __forceinline__ float unbounded_lg(float z, float escale) {
    if constexpr (Map == MAP_LOG_DECAY) return kLog2e * z;
    const float x = escale * z;
    return -(fmaxf(x, 0.f) * kLog2e + lg2_approx(1.f + ex2_approx(-fabsf(x) * kLog2e)));
}
constexpr float kPairThreshold = 7.5e-37f;   // 2^-120: below it, e^{-b} nears fp32's limit

__device__ __forceinline__ void note_timeout(volatile int *flag) {
    *flag = 1;
    atomicAdd(&g_tc_timeouts, 1u);
}

// Map: the launch's gate map; an unbounded one compiles in the per-tile
// pair path, which the bounded instance carries none of.  Split: the
// chains are the virtual sequences of a segment split (PrefillArgs::vseg);
// the plain instance carries none of that code either.  Ckpt: state
// checkpoints are written (PrefillArgs::ckpt set); without it the tile loop
// has no checkpoint test.  Shape: the gate's shape, runtime (SHAPE_ANY) or
// compiled in: one input per key channel (the default gate, eq. (5)) or one
// per (token, head), with the gate-shape tests constant.
template <int Map, bool Split, bool Ckpt, int Shape>
__global__ void __launch_bounds__(NTHREADS, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_ft,
                  const __grid_constant__ CUtensorMap tm_fz, PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + OFF_SLOT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + OFF_FLAG);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chain = blockIdx.x;
    const int n = chain / a.H, h = chain % a.H;
    int bos, eos, vflags = 0, src = n;   // src: the sequence whose init_state enters
    if constexpr (Split) {                // a virtual sequence of the segment split
        const int4 e = a.vseg[n];
        vflags = e.z;
        if (vflags & VSEG_EMPTY) return;  // uniform: the CTA has not started anything
        bos = min(max(e.x, 0), a.T_total);
        eos = min(max(e.y, bos), a.T_total);
        src = e.w;
    } else {
        seq_span(a, n, bos, eos);
    }
    // v = 0 (a transition run): the V loads address heads past H, so the
    // whole box lies outside the tensor and TMA writes its zero fill (the
    // transaction still counts the full box); no branch in the tile loop.
    const int v_head = (vflags & VSEG_ZERO_V) ? h + a.H : h;
    const int ntiles = (eos - bos + C - 1) / C;
    const size_t state_off = static_cast<size_t>(chain) * D * D;
    // gate source: a TMA tile of per-channel inputs (eq. (5)), one input per
    // (token, head) shared by the channels, or none (alpha = 1)
    const bool gate_none = Shape == SHAPE_ANY && a.gate_mode == KDA_GATE_NONE;
    const bool z_tile = Shape == SHAPE_CHANNEL || (Shape == SHAPE_ANY && !gate_none && !a.gate_scalar);
    // unbounded maps (the gate as the log-decay, Kimi Linear's -softplus):
    // a tile whose cumulative decay leaves fp32's range for e^{-b} takes the
    // position-pair path for L and A
    constexpr bool unbounded = Map != MAP_BOUNDED;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars[B_RAW + s], 1);
            mbar_init(&bars[B_FULL + s], 128);
        }
        mbar_init(&bars[B_VT], NACC + 1); // one commit per (e) issuer and the U^T issuer
        mbar_init(&bars[B_UPD], 2);       // commits of the (g) and (h) issuers
        mbar_init(&bars[B_DRAIN], 5);     // abort only: one commit per MMA-issuing thread
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    if (tid == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        if (a.gate_mode != KDA_GATE_NONE && !a.gate_scalar) prefetch_tmap(&tm_z);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
        // ------------------------------------------------------------ producers
        const int pg = (warp - 8) >> 2;     // producer warpgroup: tiles t = pg (mod 2)
        const int c = tid - NCHAIN - 128 * pg;
        const int pw = (warp - 8) & 3;
        const uint32_t pbar = 1 + 2 * pg;   // its named barrier (chain uses 2)
        const float escale = a.A_log ? expf(__ldg(a.A_log + h)) : 1.0f;
        const __nv_bfloat16 *gbeta = static_cast<const __nv_bfloat16 *>(a.beta);
        uint8_t *scr = base + OFF_SCR + pg * SCR_BYTES;
        float *kgm = reinterpret_cast<float *>(scr + SC_KGM);
        float *qgm = reinterpret_cast<float *>(scr + SC_QGM);
        float *kim = reinterpret_cast<float *>(scr + SC_KIM);
        float *ls = reinterpret_cast<float *>(scr + SC_LS);
        float *tbf = reinterpret_cast<float *>(scr + SC_TBF);
        float *t11 = reinterpret_cast<float *>(scr + SC_T11);
        float *t00 = reinterpret_cast<float *>(scr + SC_T00);
        float *ysc = reinterpret_cast<float *>(scr + SC_Y);
        // beta is a strided gather (one value per token): load it a tile ahead
        // so its latency hides behind a tile of work.
        auto load_beta = [&](int tt) {
            const int tok = bos + tt * C + c;
            return (c < C && tt < ntiles && tok < eos)
                       ? __bfloat162float(gbeta[static_cast<size_t>(tok) * a.H + h]) : 0.f;
        };
        float bt_next = load_beta(pg);
        // per-head gate: lane l < 16 of every producer warp holds row l's input, a tile ahead
        const __nv_bfloat16 *gzs = static_cast<const __nv_bfloat16 *>(a.g);
        auto load_zs = [&](int tt) {
            const int tok = bos + tt * C + lane;
            return (!z_tile && !gate_none && lane < C && tt < ntiles && tok < eos)
                       ? __bfloat162float(gzs[static_cast<size_t>(tok) * a.H + h]) : 0.f;
        };
        float zs_next = load_zs(pg);
        for (int t = pg; t < ntiles; t += NPROD) {
            const int s = t % NS;
            uint8_t *st = base + s * STAGE_BYTES;
            const int t0 = bos + t * C;
            const int nv = min(C, eos - t0);
            const float bt = bt_next;
            bt_next = load_beta(t + NPROD);
            const float zs = zs_next;
            zs_next = load_zs(t + NPROD);
            if (!mbar_wait(&bars[B_RAW + s], (t / NS) & 1, kWaitLimitNs)) note_timeout(abort_flag);
            // the abort flag as seen after this tile's own wait; read here so
            // its latency is off the barrier that publishes it
            const bool abort_seen = *abort_flag != 0;

            // Gate and decays in log2 units, branch-free: the retention
            // a_r = 2^{g_r / ln 2}; prefix products give e^{b_r}, suffix
            // products e^{b_C - b_r}, and e^{-b_r} = e^{b_C - b_r} / e^{b_C}.
            // Thread (cp, hh) owns channels c0, c0 + 1 of rows 8 hh .. 8 hh + 7;
            // the two row halves (lanes l, l ^ 16) join their products by shuffle.
            const int cp = lane & 15, hh = lane >> 4;
            const int c0 = 32 * pw + 2 * cp;
            // (channel c0, channel c0 + 1) pairs, packed for the f32x2 pipe
            f32x2 kx[8], qx[8], pre[8], suf[8];
            if (z_tile && !unbounded) {                 // eq. (5) per key channel
                const f32x2 zc = pack2(-kLog2e * escale, -kLog2e * escale);
                const f32x2 lc = pack2(kLog2e * a.g_min, kLog2e * a.g_min);
                const f32x2 one = pack2(1.f, 1.f);
                // full tiles (all but a sequence's last) without the row masks
                auto gate_rows = [&](auto full) {
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int row = 8 * hh + r;
                        const bool in = decltype(full)::value || row < nv;
                        const uint32_t zz = *reinterpret_cast<const uint32_t *>(st + ST_Z + row * 256 + c0 * 2);
                        const uint32_t kk = in ? *reinterpret_cast<const uint32_t *>(st + ST_K + row * 256 + c0 * 2) : 0u;
                        const uint32_t qq = in ? *reinterpret_cast<const uint32_t *>(st + ST_Q + row * 256 + c0 * 2) : 0u;
                        kx[r] = pack2(bf16_half(kk, 0), bf16_half(kk, 1));
                        qx[r] = pack2(bf16_half(qq, 0), bf16_half(qq, 1));
                        const float2 e = unpack2(fmul2(zc, pack2(bf16_half(zz, 0), bf16_half(zz, 1))));
                        const f32x2 den = fadd2(one, pack2(ex2_approx(e.x), ex2_approx(e.y)));
                        const float2 lg = unpack2(fmul2(lc, pack2(rcp_approx(unpack2(den).x), rcp_approx(unpack2(den).y))));
                        suf[r] = in ? pack2(ex2_approx(lg.x), ex2_approx(lg.y)) : one;   // a_r (1 past the end)
                    }
                };
                if (nv == C) gate_rows(std::true_type{});
                else gate_rows(std::false_type{});
            } else if (z_tile) {                        // unbounded map per key channel
                // full tiles without the row masks, as for the bounded map
                auto gate_rows = [&](auto full) {
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int row = 8 * hh + r;
                        const bool in = decltype(full)::value || row < nv;
                        const uint32_t zz = *reinterpret_cast<const uint32_t *>(st + ST_Z + row * 256 + c0 * 2);
                        const uint32_t kk = in ? *reinterpret_cast<const uint32_t *>(st + ST_K + row * 256 + c0 * 2) : 0u;
                        const uint32_t qq = in ? *reinterpret_cast<const uint32_t *>(st + ST_Q + row * 256 + c0 * 2) : 0u;
                        kx[r] = pack2(bf16_half(kk, 0), bf16_half(kk, 1));
                        qx[r] = pack2(bf16_half(qq, 0), bf16_half(qq, 1));
                        suf[r] = in ? pack2(ex2_approx(unbounded_lg<Map>(bf16_half(zz, 0), escale)),
                                            ex2_approx(unbounded_lg<Map>(bf16_half(zz, 1), escale)))
                                    : pack2(1.f, 1.f);
                    }
                };
                if (nv == C) gate_rows(std::true_type{});
                else gate_rows(std::false_type{});
            } else {                                    // one gate per (token, head), or none
                auto gate_rows = [&](auto full) {
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int row = 8 * hh + r;
                        const bool in = decltype(full)::value || row < nv;
                        const uint32_t kk = in ? *reinterpret_cast<const uint32_t *>(st + ST_K + row * 256 + c0 * 2) : 0u;
                        const uint32_t qq = in ? *reinterpret_cast<const uint32_t *>(st + ST_Q + row * 256 + c0 * 2) : 0u;
                        const float z = __shfl_sync(0xffffffffu, zs, row);
                        float lg;
                        if (unbounded) {
                            lg = unbounded_lg<Map>(z, escale);
                        } else {
                            const float sig = rcp_approx(1.f + ex2_approx(-kLog2e * escale * z));
                            lg = gate_none ? 0.f : (kLog2e * a.g_min) * sig;
                        }
                        const float a_r = in ? ex2_approx(lg) : 1.f;
                        kx[r] = pack2(bf16_half(kk, 0), bf16_half(kk, 1));
                        qx[r] = pack2(bf16_half(qq, 0), bf16_half(qq, 1));
                        suf[r] = pack2(a_r, a_r);
                    }
                };
                // full tiles without the row masks only where the shape is compiled in
                if (Shape == SHAPE_HEAD && nv == C) gate_rows(std::true_type{});
                else gate_rows(std::false_type{});
            }
            float gC[2], inv_gC[2];
            {
                f32x2 run = pack2(1.f, 1.f);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    run = fmul2(run, suf[r]);
                    pre[r] = run;
                }
                const float2 rr = unpack2(run);
                const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, rr.x, 16),   // the other half's
                                                 __shfl_xor_sync(0xffffffffu, rr.y, 16));  // products
                const f32x2 oth = pack2(other.x, other.y);
                const float2 g2 = unpack2(fmul2(run, oth));                             // e^{b_C}
                gC[0] = g2.x; gC[1] = g2.y;
                const f32x2 one = pack2(1.f, 1.f);
                const f32x2 lead = hh ? oth : one;                                       // decay before this half
                f32x2 back = hh ? one : oth;                                             // decay after this half
#pragma unroll
                for (int r = 7; r >= 0; --r) {
                    const f32x2 a_r = suf[r];
                    suf[r] = back;                                                       // e^{b_C - b_r}
                    back = fmul2(back, a_r);
                    pre[r] = fmul2(pre[r], lead);                                        // e^{b_r}
                }
                inv_gC[0] = rcp_approx(gC[0]);
                inv_gC[1] = rcp_approx(gC[1]);
            }
            if (hh == 0) *reinterpret_cast<float2 *>(st + ST_GC + c0 * 4) = make_float2(gC[0], gC[1]);
            if (c < C) reinterpret_cast<float *>(st + ST_BETA)[c] = bt;
            const f32x2 igc = pack2(inv_gC[0], inv_gC[1]);
            // 128B-swizzled offsets of this thread's rows: row 0's offset has
            // zeros in bits 4-9, so row r's is it XOR (r << 7 | r << 4)
            const uint32_t wq0 = off_kmajor_sw128(16 + 8 * hh, c0, 32);
            const uint32_t kd0 = off_mnmajor_sw128(c0, 8 * hh, C);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int row = 8 * hh + r;
                const uint32_t sw = static_cast<uint32_t>((r << 7) | (r << 4));
                const float2 kg = unpack2(fmul2(kx[r], pre[r]));
                const float2 qg = unpack2(fmul2(qx[r], pre[r]));
                const f32x2 kd2 = fmul2(kx[r], suf[r]);
                const float2 kd = unpack2(kd2);
                const float2 ki = unpack2(fmul2(kd2, igc));
                *reinterpret_cast<uint32_t *>(st + ST_WQ + (wq0 ^ sw)) = pack_h2(qg.x, qg.y);
                *reinterpret_cast<uint32_t *>(st + ST_KD + (kd0 ^ sw)) = pack_h2(kd.x, kd.y);
                *reinterpret_cast<float2 *>(qgm + row * PADF + c0) = make_float2(tf32_operand(qg.x), tf32_operand(qg.y));
                *reinterpret_cast<float2 *>(kgm + row * PADF + c0) = make_float2(tf32_operand(kg.x), tf32_operand(kg.y));
                *reinterpret_cast<float2 *>(kim + row * PADF + c0) = make_float2(tf32_operand(ki.x), tf32_operand(ki.y));
            }
            if (named_bar_or(pbar, 128, abort_seen)) break;   // uniform across the warpgroup
            const bool pair_tile =
                unbounded && named_bar_or(pbar, 128, gC[0] < kPairThreshold || gC[1] < kPairThreshold);

            if constexpr (unbounded) if (pair_tile) {
                // L_ri = sum_c k_rc k_ic 2^{B_rc - B_ic}, A_ri = sum_c q_rc k_ic 2^{B_rc - B_ic}
                // (i <= r, so every exponent is <= 0), B the in-tile cumulative
                // log2-decay, stored in the K e^-b operand's place.
                float bv[2][8], cum[2] = {0.f, 0.f};
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int row = 8 * hh + r;
                    const float m = row < nv ? 1.f : 0.f;
                    const uint32_t zz = z_tile ? *reinterpret_cast<const uint32_t *>(st + ST_Z + row * 256 + c0 * 2) : 0u;
                    const float zr = __shfl_sync(0xffffffffu, zs, row);
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        cum[ch] += m * unbounded_lg<Map>(z_tile ? bf16_half(zz, ch) : zr, escale);
                        bv[ch][r] = cum[ch];
                    }
                }
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const float other = __shfl_xor_sync(0xffffffffu, cum[ch], 16);
                    const float lead = hh ? other : 0.f;
#pragma unroll
                    for (int r = 0; r < 8; ++r) kim[(8 * hh + r) * PADF + c0 + ch] = bv[ch][r] + lead;
                }
                named_bar_sync(pbar, 128);
#pragma unroll 1
                for (int pass = 0; pass < 2; ++pass) {
                    const int e = c + 128 * pass;
                    const int r = e >> 4, i = e & 15;
                    float l = 0.f, aa = 0.f;
                    if (i <= r && r < nv) {
                        const float *br = kim + r * PADF, *bi = kim + i * PADF;
#pragma unroll 4
                        for (int jj = 0; jj < D; ++jj) {
                            const int ch = (lane + jj) & (D - 1);   // rotated start: distinct banks
                            const float ki = bf16_at(st + ST_K + i * 256 + ch * 2) * ex2_approx(br[ch] - bi[ch]);
                            l = fmaf(bf16_at(st + ST_K + r * 256 + ch * 2), ki, l);
                            aa = fmaf(bf16_at(st + ST_Q + r * 256 + ch * 2), ki, aa);
                        }
                    }
                    ls[r * LSS + i] = i < r ? l : 0.f;
                    st_h(st + ST_AT + off_kmajor_none(r, i, C), i <= r ? aa : 0.f);
                }
            }
            if (!pair_tile) {
                // one 16x8 block per warp: pw 0/1 -> L columns 0-7/8-15, pw 2/3 -> A
                const int g = lane >> 2, tq = lane & 3;
                const float *lhs = pw < 2 ? kgm : qgm;
                const int n0 = (pw & 1) * 8;
                float d4[4] = {0.f, 0.f, 0.f, 0.f}, d4b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k0 = 0; k0 < D; k0 += 16) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int kb = k0 + 8 * hh;
                        const uint32_t a0 = __float_as_uint(lhs[g * PADF + kb + tq]);
                        const uint32_t a1 = __float_as_uint(lhs[(g + 8) * PADF + kb + tq]);
                        const uint32_t a2 = __float_as_uint(lhs[g * PADF + kb + tq + 4]);
                        const uint32_t a3 = __float_as_uint(lhs[(g + 8) * PADF + kb + tq + 4]);
                        const uint32_t b0 = __float_as_uint(kim[(n0 + g) * PADF + kb + tq]);
                        const uint32_t b1 = __float_as_uint(kim[(n0 + g) * PADF + kb + tq + 4]);
                        mma_1688_tf32(hh ? d4b : d4, a0, a1, a2, a3, b0, b1);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) d4[e] += d4b[e];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = g + (e >> 1) * 8;
                    const int col = n0 + 2 * tq + (e & 1);
                    if (pw < 2)
                        ls[row * LSS + col] = col < row ? d4[e] : 0.f;
                    else
                        st_h(st + ST_AT + off_kmajor_none(row, col, C), col <= row ? d4[e] : 0.f);
                }
            }
            named_bar_sync(pbar, 128);
            // T = (I + N)^-1, N = Diag(beta) L strictly lower, in 8x8 blocks:
            // T00 = (I + N00)^-1 and T11 = (I + N11)^-1 by forward substitution
            // (lanes 0-7 / 8-15 of the first warp own one column each, right-
            // looking: once x_m is final every later x_i loses N_im x_m, so the
            // dependent chain is one FMA per step), then T10 = -T11 (N10 T00) as
            // two 8x8 products over the same warp.  Stored as T Diag(beta),
            // tf32-rounded.  Only warp 0 works; one barrier follows.
            const float *betas = reinterpret_cast<const float *>(st + ST_BETA);
            auto row8 = [&](const float *p, float (&x)[8]) {   // 8 floats, two 16-byte loads
                const float4 lo = *reinterpret_cast<const float4 *>(p);
                const float4 hi = *reinterpret_cast<const float4 *>(p + 4);
                x[0] = lo.x; x[1] = lo.y; x[2] = lo.z; x[3] = lo.w;
                x[4] = hi.x; x[5] = hi.y; x[6] = hi.z; x[7] = hi.w;
            };
            if (pw == 0) {
                if (lane < C) {
                    const int j = lane, blk = j >> 3, r0 = 8 * blk;
                    float br[8], lr[8][8];
                    row8(betas + r0, br);
#pragma unroll
                    for (int i = 1; i < 8; ++i) row8(ls + (r0 + i) * LSS + r0, lr[i]);
                    float x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = r0 + i == j ? 1.f : 0.f;
#pragma unroll
                    for (int m = 0; m < 7; ++m)
#pragma unroll
                        for (int i = m + 1; i < 8; ++i) x[i] = fmaf(-br[i] * lr[i][m], x[m], x[i]);
                    const float bj = betas[j];
                    float *tdiag = blk ? t11 : t00;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        tdiag[i * 8 + (j - r0)] = x[i];
                        tbf[(r0 + i) * TBS + j] = to_tf32(x[i] * bj);
                        if (blk) tbf[i * TBS + j] = 0.f;           // T01 = 0
                    }
                }
                __syncwarp();
                // Y = Diag(beta_8..15) L10 T00 and T10 = -T11 Y: two entries per lane
                float yv[2];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int e = lane + 32 * h2, bi = e >> 3, bj8 = e & 7;
                    float lr[8];
                    row8(ls + (8 + bi) * LSS, lr);
                    float acc = 0.f;
#pragma unroll
                    for (int m2 = 0; m2 < 8; ++m2) acc = fmaf(lr[m2], t00[m2 * 8 + bj8], acc);
                    yv[h2] = betas[8 + bi] * acc;
                }
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) ysc[lane + 32 * h2] = yv[h2];
                __syncwarp();
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int e = lane + 32 * h2, bi = e >> 3, bj8 = e & 7;
                    float tr[8];
                    row8(t11 + bi * 8, tr);
                    float acc = 0.f;
#pragma unroll
                    for (int m2 = 0; m2 < 8; ++m2) acc = fmaf(tr[m2], ysc[m2 * 8 + bj8], acc);
                    tbf[(8 + bi) * TBS + bj8] = to_tf32(-acc * betas[bj8]);
                }
            }
            named_bar_sync(pbar, 128);
            // T Diag(beta) as the bf16 B operand of U^T = V^T (T Diag(beta))^T
            // (a tcgen05 product the chain issues): hi + lo reproduce the
            // tf32-rounded values exactly (at most 11 significant bits).
            {
                const int r = c >> 3, i0 = 2 * (c & 7);
                const uint32_t off = (r >> 3) * 256 + (i0 >> 3) * 128 + (r & 7) * 16 + (i0 & 7) * 2;
                const float x0 = tbf[r * TBS + i0], x1 = tbf[r * TBS + i0 + 1];
                const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
                const __nv_bfloat162 lo = __floats2bfloat162_rn(x0 - __low2float(hi), x1 - __high2float(hi));
                *reinterpret_cast<__nv_bfloat162 *>(st + ST_TB + off) = hi;
                *reinterpret_cast<__nv_bfloat162 *>(st + ST_TB + 512 + off) = lo;
            }
            // W = T Diag(beta) (K e^b) -> rows 0..15 of the (e) B operand hold -W.
            // 16 x 16 x 128, tf32 mma.sync; warp pw covers channels [32 pw, 32 pw + 32).
            {
                const int g = lane >> 2, tq = lane & 3;
                uint32_t ta[2][4];
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int k0 = ks * 8;
                    ta[ks][0] = __float_as_uint(tbf[g * TBS + k0 + tq]);
                    ta[ks][1] = __float_as_uint(tbf[(g + 8) * TBS + k0 + tq]);
                    ta[ks][2] = __float_as_uint(tbf[g * TBS + k0 + tq + 4]);
                    ta[ks][3] = __float_as_uint(tbf[(g + 8) * TBS + k0 + tq + 4]);
                }
                // n index n of n-block nb is channel 32 pw + 4 n + nb: a lane's B
                // fragments for the four n-blocks are one float4, and its output
                // columns (n = 2 tq, 2 tq + 1) are channels 32 pw + 8 tq + 0..7.
                float dw[4][4];
#pragma unroll
                for (int nb = 0; nb < 4; ++nb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) dw[nb][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int s0 = ks * 8 + tq;
                    const float4 b0 = *reinterpret_cast<const float4 *>(kgm + s0 * PADF + pw * 32 + 4 * g);
                    const float4 b1 = *reinterpret_cast<const float4 *>(kgm + (s0 + 4) * PADF + pw * 32 + 4 * g);
                    const float bl0[4] = {b0.x, b0.y, b0.z, b0.w}, bl1[4] = {b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                    for (int nb = 0; nb < 4; ++nb)
                        mma_1688_tf32(dw[nb], ta[ks][0], ta[ks][1], ta[ks][2], ta[ks][3], __float_as_uint(bl0[nb]),
                                      __float_as_uint(bl1[nb]));
                }
                // channel 32 pw + 8 tq + nb <- dw[nb][0 | 2], + 4 + nb <- dw[nb][1 | 3]
                const int c0 = pw * 32 + 8 * tq;
                const uint4 w_lo = make_uint4(pack_h2(-dw[0][0], -dw[1][0]), pack_h2(-dw[2][0], -dw[3][0]),
                                              pack_h2(-dw[0][1], -dw[1][1]), pack_h2(-dw[2][1], -dw[3][1]));
                const uint4 w_hi = make_uint4(pack_h2(-dw[0][2], -dw[1][2]), pack_h2(-dw[2][2], -dw[3][2]),
                                              pack_h2(-dw[0][3], -dw[1][3]), pack_h2(-dw[2][3], -dw[3][3]));
                *reinterpret_cast<uint4 *>(st + ST_WQ + off_kmajor_sw128(g, c0, 32)) = w_lo;
                *reinterpret_cast<uint4 *>(st + ST_WQ + off_kmajor_sw128(g + 8, c0, 32)) = w_hi;
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_FULL + s]);
        }
    } else {
        // ------------------------------------------------------------ chain
        const int j = tid & 127;           // value channel = TMEM lane
        const int hf = tid >> 7;           // which half of the key rows / tile columns
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const long long ck_row0 = Ckpt ? ckpt_first_row(a, n) : 0;
        constexpr int HR = D / 2;          // state rows per thread
        constexpr uint32_t id_e = idesc_f16kind(kTypeF16, 128, 32, 0, 0);
        constexpr uint32_t id_g = idesc_f16kind(kTypeF16, 128, 16, 0, 0);
        constexpr uint32_t id_h = idesc_f16kind(kTypeF16, 128, 128, 0, 1);
        const uint32_t sb = smem_u32(base);
        // TMA loads of tile tt into its ring stage (one thread).
        auto issue_tma = [&](int tt) {
            const int ss = tt % NS;
            uint8_t *stg = base + ss * STAGE_BYTES;
            const int tok = bos + tt * C;
            mbar_arrive_expect_tx(&bars[B_RAW + ss], z_tile ? TX_BYTES : TX_BYTES_NOZ);
            tma_load_3d(stg + ST_Q, &tm_q, &bars[B_RAW + ss], 0, h, tok);
            tma_load_3d(stg + ST_K, &tm_k, &bars[B_RAW + ss], 0, h, tok);
            if (z_tile) tma_load_3d(stg + ST_Z, &tm_z, &bars[B_RAW + ss], 0, h, tok);
            tma_load_3d(stg + ST_V, &tm_v, &bars[B_RAW + ss], 0, v_head, tok);          // channels 0-63
            tma_load_3d(stg + ST_V + 2048, &tm_v, &bars[B_RAW + ss], 64, v_head, tok);  // channels 64-127
        };
        constexpr int TMA_TID = 160, OST_TID = 192;  // lane 0 of chain warps 5 and 6
        int tma_next = 0;                            // (TMA thread) next tile to load
        if (tid == TMA_TID)
            for (; tma_next < NS && tma_next < ntiles; ++tma_next) issue_tma(tma_next);
        // (e) for tile tt: issuer p (lane 0 of chain warp p) issues the K slices
        // p and p + 4 into accumulator p once the tile's operands are ready.
        auto issue_e = [&](int tt, int p) -> bool {
            const int ss = tt % NS;
            if (!mbar_wait(&bars[B_FULL + ss], (tt / NS) & 1, kWaitLimitNs)) return false;
            tc_fence_after();
            const uint32_t st = sb + ss * STAGE_BYTES;
            const uint32_t e_acc = tmem + TM_E + E_BUF * static_cast<uint32_t>(tt & 1) + 32u * p;
#pragma unroll
            for (int h2 = 0; h2 < D / 16 / NACC; ++h2) {
                const int kk = p + NACC * h2;
                const int k = kk * 16;
                const uint32_t b_off = ST_WQ + (k >> 6) * (32 * 128) + (k & 63) * 2;
                mma_f16kind_tmem_a(e_acc, tmem + TM_ST + 8 * kk, smem_desc(st + b_off, 16, 1024, kLayoutSW128),
                                   id_e, h2 > 0 ? 1u : 0u);
            }
            mma_commit(&bars[B_VT]);
            return true;
        };
        const bool e_issuer = lane == 0 && warp < NACC;   // chain warps 0..3, lane 0
        // U^T = V^T (T Diag(beta))^T for tile tt into slot tt & 1 (two bf16
        // products, hi then lo part of T Diag(beta)), committed with (e).
        constexpr int U_TID = 224;                        // lane 0 of chain warp 7
        constexpr uint32_t id_u = idesc_f16kind(kTypeBF16, 128, 16, 1, 0);
        auto issue_u = [&](int tt) -> bool {
            const int ss = tt % NS;
            if (!mbar_wait(&bars[B_FULL + ss], (tt / NS) & 1, kWaitLimitNs)) return false;
            tc_fence_after();
            const uint32_t st = sb + ss * STAGE_BYTES;
            const uint64_t av = smem_desc(st + ST_V, 2048, 1024, kLayoutSW128);
            const uint32_t d = tmem + TM_U + 16u * static_cast<uint32_t>(tt & 1);
            mma_f16kind(d, av, smem_desc(st + ST_TB, 128, 256, kLayoutNone), id_u, 0);
            mma_f16kind(d, av, smem_desc(st + ST_TB + 512, 128, 256, kLayoutNone), id_u, 1);
            mma_commit(&bars[B_VT]);
            return true;
        };

        float S[HR];
        if constexpr (Split) {
            const size_t init_off = (static_cast<size_t>(src) * a.H + h) * D * D;
            const bool init_given = a.init_state && !(vflags & (VSEG_ZERO_INIT | VSEG_IDENT_INIT));
#pragma unroll
            for (int cc = 0; cc < HR; ++cc)
                S[cc] = (vflags & VSEG_IDENT_INIT) ? (hf * HR + cc == j ? 1.f : 0.f)
                        : init_given ? a.init_state[init_off + static_cast<size_t>(hf * HR + cc) * D + j] : 0.f;
        } else {
#pragma unroll
            for (int cc = 0; cc < HR; ++cc)
                S[cc] = a.init_state ? a.init_state[state_off + static_cast<size_t>(hf * HR + cc) * D + j] : 0.f;
        }
        // fp16 S^T row j, K range [64 hf, 64 hf + 64) -> 32 TMEM columns
        auto write_sT = [&]() {
            uint32_t pk[HR / 2];
#pragma unroll
            for (int i = 0; i < HR / 2; ++i) pk[i] = pack_h2(S[2 * i], S[2 * i + 1]);
            tmem_st32(tmem + TM_ST + lane_base + hf * (HR / 2), pk);
            tmem_st_wait();
        };
        write_sT();
        tc_fence_before();
        named_bar_sync(2, NCHAIN);
        if (e_issuer && ntiles > 0 && !issue_e(0, warp)) note_timeout(abort_flag);
        if (tid == U_TID && ntiles > 0 && !issue_u(0)) note_timeout(abort_flag);

        __nv_bfloat16 *gout = static_cast<__nv_bfloat16 *>(a.out);
        // every run of a segment split writes fp32 rows, unrounded, to
        // out_trans or out_zero (by its flags; the same code for every run)
        const bool f_trans = (vflags & VSEG_OUT_TRANS) != 0;
        uint8_t *ost = base + OFF_OST;
        // O of tile tt, rows [8 hf, 8 hf + 8): sum of the accumulators' columns
        // 16..31.  Full tiles go to a staging tile stored by TMA (bf16: two
        // tiles, alternating; fp32: one tile, the whole staging area, free
        // again before the next chain barrier), a sequence's partial last tile
        // straight to global memory.
        auto read_out = [&](int tt) {
            const uint32_t eb = tmem + TM_E + E_BUF * static_cast<uint32_t>(tt & 1) + lane_base + 16 + 8 * hf;
            float o[8], x[NACC - 1][8];
            tmem_ld8(eb, o);
#pragma unroll
            for (int p = 1; p < NACC; ++p) tmem_ld8(eb + 32u * p, x[p - 1]);
            tmem_ld_wait();
#pragma unroll
            for (int p = 1; p < NACC; ++p)
#pragma unroll
                for (int r = 0; r < 8; r += 2) {
                    const float2 y = unpack2(fadd2(pack2(o[r], o[r + 1]), pack2(x[p - 1][r], x[p - 1][r + 1])));
                    o[r] = y.x; o[r + 1] = y.y;
                }
            const int tt0 = bos + tt * C;
            const int nvv = min(C, eos - tt0);
            if (Split && nvv == C) {
                float *stg = reinterpret_cast<float *>(ost);
#pragma unroll
                for (int r = 0; r < 8; ++r) stg[(8 * hf + r) * D + j] = a.scale * o[r];
                fence_proxy_async_smem();
            } else if constexpr (Split) {
                float *op = (f_trans ? a.out_trans : a.out_zero) + static_cast<size_t>(tt0 + 8 * hf) * a.H * D + static_cast<size_t>(h) * D + j;
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (8 * hf + r < nvv) op[static_cast<size_t>(r) * a.H * D] = a.scale * o[r];
            } else if (nvv == C) {
                __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(ost + (tt & 1) * (C * D * 2));
                const f32x2 sc = pack2(a.scale, a.scale);
#pragma unroll
                for (int r = 0; r < 8; r += 2) {
                    const float2 y = unpack2(fmul2(pack2(o[r], o[r + 1]), sc));
                    stg[(8 * hf + r) * D + j] = __float2bfloat16_rn(y.x);
                    stg[(8 * hf + r + 1) * D + j] = __float2bfloat16_rn(y.y);
                }
                fence_proxy_async_smem();
            } else {
                __nv_bfloat16 *op = gout + static_cast<size_t>(tt0 + 8 * hf) * a.H * D + static_cast<size_t>(h) * D + j;
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (8 * hf + r < nvv) op[static_cast<size_t>(r) * a.H * D] = __float2bfloat16_rn(a.scale * o[r]);
            }
        };
        // after a chain barrier that follows read_out(tt): one thread stores the staged tile
        auto store_out = [&](int tt) {
            const int tt0 = bos + tt * C;
            if (min(C, eos - tt0) == C) {
                if constexpr (Split) tma_store_3d(f_trans ? &tm_ft : &tm_fz, ost, 0, h, tt0);
                else tma_store_3d(&tm_o, ost + (tt & 1) * (C * D * 2), 0, h, tt0);
                bulk_commit();
            }
            if constexpr (!Split) bulk_wait_read<1>();   // the other staging tile is free again
        };
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % NS;
            const uint8_t *st = base + s * STAGE_BYTES;
            const uint32_t e_acc = tmem + TM_E + E_BUF * static_cast<uint32_t>(t & 1);
            bool ok = mbar_wait(&bars[B_VT], t & 1, kWaitLimitNs);
            ok = mbar_wait(&bars[B_FULL + s], (t / NS) & 1, kWaitLimitNs) && ok;   // U, e^{b_C} visible
            if (!ok) note_timeout(abort_flag);
            const bool abort_seen = *abort_flag != 0;   // read early: off the barrier below
            tc_fence_after();
            {
                // tile columns [8 hf, 8 hf + 8) of Vt^T = U^T - (W S)^T
                float uj[8], v[NACC][8];
#pragma unroll
                for (int p = 0; p < NACC; ++p) tmem_ld8(e_acc + 32u * p + lane_base + 8 * hf, v[p]);
                tmem_ld8(tmem + TM_U + 16u * static_cast<uint32_t>(t & 1) + lane_base + 8 * hf, uj);
                tmem_ld_wait();
#pragma unroll
                for (int p = 0; p < NACC; ++p)
#pragma unroll
                    for (int r = 0; r < 8; r += 2) {
                        const float2 x = unpack2(fadd2(pack2(uj[r], uj[r + 1]), pack2(v[p][r], v[p][r + 1])));
                        uj[r] = x.x; uj[r + 1] = x.y;
                    }
                uint32_t p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) p[i] = pack_h2(uj[2 * i], uj[2 * i + 1]);
                tmem_st4(tmem + TM_VT + lane_base + 4 * hf, p);
                tmem_st_wait();
            }
            tc_fence_before();
            // fp32 staging: the previous tile's store has read it before the
            // chain passes this barrier (read_out writes it next)
            if constexpr (Split) if (tid == OST_TID) bulk_wait_read<0>();
            if (named_bar_or(2, NCHAIN, abort_seen)) break;   // uniform across the chain
            if (lane == 0 && warp < 2) {
                tc_fence_after();
                const uint32_t stb = sb + s * STAGE_BYTES;
                if (warp == 0)      // (g) E[:,16:32] += Vt^T A^T
                    mma_f16kind_tmem_a(e_acc + 16, tmem + TM_VT, smem_desc(stb + ST_AT, 128, 256, kLayoutNone),
                                       id_g, 1);
                else                // (h) H = Vt^T (K e^{b_C - b})
                    mma_f16kind_tmem_a(tmem + TM_H, tmem + TM_VT, smem_desc(stb + ST_KD, 2048, 1024, kLayoutSW128),
                                       id_h, 0);
                mma_commit(&bars[B_UPD]);
            }
            if (t > 0) read_out(t - 1);    // overlaps (g)/(h)
            if (!mbar_wait(&bars[B_UPD], t & 1, kWaitLimitNs)) note_timeout(abort_flag);
            tc_fence_after();
            const float *gc = reinterpret_cast<const float *>(st + ST_GC) + hf * HR;
#pragma unroll
            for (int cb = 0; cb < HR / 16; cb += 2) {      // two TMEM loads per wait
                float inc[2][16];
                tmem_ld16(tmem + TM_H + lane_base + hf * HR + cb * 16, inc[0]);
                tmem_ld16(tmem + TM_H + lane_base + hf * HR + cb * 16 + 16, inc[1]);
                tmem_ld_wait();
#pragma unroll
                for (int b2 = 0; b2 < 2; ++b2) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {   // e^{b_C}: the same 16 values for the whole warp
                        const float4 g4 = *reinterpret_cast<const float4 *>(gc + (cb + b2) * 16 + q4 * 4);
                        float *sp = S + (cb + b2) * 16 + q4 * 4;
                        const float *ip = inc[b2] + q4 * 4;
                        const float2 lo = unpack2(ffma2(pack2(g4.x, g4.y), pack2(sp[0], sp[1]), pack2(ip[0], ip[1])));
                        const float2 hi = unpack2(ffma2(pack2(g4.z, g4.w), pack2(sp[2], sp[3]), pack2(ip[2], ip[3])));
                        sp[0] = lo.x; sp[1] = lo.y; sp[2] = hi.x; sp[3] = hi.y;
                    }
                }
            }
            write_sT();
            tc_fence_before();
            named_bar_sync(2, NCHAIN);   // (the abort flag is polled once a tile, at the Vt barrier)
            // every read of this stage (TMA tiles, U, e^{b_C}, MMA operands) is done
            if (e_issuer && t + 1 < ntiles && !issue_e(t + 1, warp)) note_timeout(abort_flag);
            if (tid == U_TID && t + 1 < ntiles && !issue_u(t + 1)) note_timeout(abort_flag);
            if (tid == TMA_TID && t + NS < ntiles) issue_tma(tma_next++);
            if (tid == OST_TID && t > 0) store_out(t - 1);
            // state checkpoint after this tile (off the chain's critical path)
            if constexpr (Ckpt) {
                if (float *cp = ckpt_slot(a, ck_row0, min((t + 1) * C, eos - bos), h, D * D)) {
#pragma unroll
                    for (int cc = 0; cc < HR; ++cc) __stcs(cp + static_cast<size_t>(hf * HR + cc) * D + j, S[cc]);
                }
            }
        }
        // uniform decision: every chain thread takes the same branch
        if constexpr (Split) if (tid == OST_TID) bulk_wait_read<0>();
        const bool aborted = named_bar_or(2, NCHAIN, *abort_flag != 0);
        if (ntiles > 0 && !aborted) {
            read_out(ntiles - 1);
            named_bar_sync(2, NCHAIN);
            if (tid == OST_TID) store_out(ntiles - 1);
        }
        if (tid == OST_TID) bulk_wait_all();
        if (aborted) {
            // A wait gave up: before the CTA frees its tensor memory and exits,
            // let the asynchronous work it started finish (bounded waits).
            //  - TMA loads: the last tile issued into each ring stage.
            //  - tcgen05 products: every MMA-issuing thread (lane 0 of chain
            //    warps 0-3: (e), (g), (h); lane 0 of warp 7: U) commits once
            //    more; the commit arrives when all its earlier products are done.
            if (tid == TMA_TID)
                for (int tt = max(0, tma_next - NS); tt < tma_next; ++tt)
                    mbar_wait(&bars[B_RAW + tt % NS], (tt / NS) & 1, kWaitLimitNs);
            if (lane == 0 && (warp < NACC || tid == U_TID)) {
                mma_commit(&bars[B_DRAIN]);
                mbar_wait(&bars[B_DRAIN], 0, kWaitLimitNs);
            }
        }
        if (a.final_state && !aborted) {
#pragma unroll
            for (int cc = 0; cc < HR; ++cc)
                a.final_state[state_off + static_cast<size_t>(hf * HR + cc) * D + j] = S[cc];
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// [T_total, H, 128] bf16 (or fp32) viewed as a 3-D tensor (d, head, token).
bool make_map(CUtensorMap *m, const void *ptr, int H, int T_total, int box_d, bool swizzle128,
              bool fp32 = false) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t esz = fp32 ? 4 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T_total)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esz, static_cast<cuuint64_t>(H) * D * esz};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_d), 1, static_cast<cuuint32_t>(C)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                           const_cast<void *>(ptr), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(kda_dtype dt, int dk, int dv) { return dt == KDA_BF16 && dk == D && dv == D; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s) {
    CUtensorMap tq, tk, tz, tv, to, tft, tfz;
    // the gate tile map exists only for per-channel gates (a per-head g_raw is
    // [T, H]; with no gate it may be NULL) -- the same test as the kernel's
    const bool z_tile = a.gate_mode != KDA_GATE_NONE && !a.gate_scalar;
    if (!make_map(&tq, a.q, a.H, a.T_total, D, false) || !make_map(&tk, a.k, a.H, a.T_total, D, false) ||
        !make_map(&tz, z_tile ? a.g : a.q, a.H, a.T_total, D, false) ||
        !make_map(&tv, a.v ? a.v : a.q, a.H, a.T_total, D / 2, true) ||
        !make_map(&to, a.out, a.H, a.T_total, D, false))
        return cudaErrorInvalidValue;
    // a segment split's fp32 row buffers (the plain kernel never reads these)
    if (a.vseg ? !make_map(&tft, a.out_trans, a.H, a.T_total, D, false, true) ||
                     !make_map(&tfz, a.out_zero, a.H, a.T_total, D, false, true)
               : false)
        return cudaErrorInvalidValue;
    if (!a.vseg) tft = tfz = to;
    const bool unbounded = a.gate_mode == KDA_GATE_LOG_DECAY || a.gate_mode == KDA_GATE_NEG_SOFTPLUS;
    const bool channel_gate = !unbounded && a.gate_mode == KDA_GATE_BOUNDED && !a.gate_scalar;
    const bool head_gate = !unbounded && a.gate_mode == KDA_GATE_BOUNDED && a.gate_scalar;
    // instance <gate map, split, checkpoints, default gate>
    using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                          CUtensorMap, PrefillArgs);
    Kern kern;
    if (unbounded) {
        const bool ld = a.gate_mode == KDA_GATE_LOG_DECAY;
        kern = a.vseg   ? (ld ? prefill_tc_kernel<MAP_LOG_DECAY, true, false, SHAPE_ANY>
                              : prefill_tc_kernel<MAP_NEG_SOFTPLUS, true, false, SHAPE_ANY>)
               : a.ckpt ? (ld ? prefill_tc_kernel<MAP_LOG_DECAY, false, true, SHAPE_ANY>
                              : prefill_tc_kernel<MAP_NEG_SOFTPLUS, false, true, SHAPE_ANY>)
                        : (ld ? prefill_tc_kernel<MAP_LOG_DECAY, false, false, SHAPE_ANY>
                              : prefill_tc_kernel<MAP_NEG_SOFTPLUS, false, false, SHAPE_ANY>);
    } else {
        kern = a.vseg   ? (channel_gate ? prefill_tc_kernel<MAP_BOUNDED, true, false, SHAPE_CHANNEL>
                                        : prefill_tc_kernel<MAP_BOUNDED, true, false, SHAPE_ANY>)
               : a.ckpt ? prefill_tc_kernel<MAP_BOUNDED, false, true, SHAPE_ANY>
               : channel_gate ? prefill_tc_kernel<MAP_BOUNDED, false, false, SHAPE_CHANNEL>
               : head_gate    ? prefill_tc_kernel<MAP_BOUNDED, false, false, SHAPE_HEAD>
                              : prefill_tc_kernel<MAP_BOUNDED, false, false, SHAPE_ANY>;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(a.N) * static_cast<unsigned>(a.H));
    kern<<<grid, NTHREADS, SMEM_BYTES, s>>>(tq, tk, tz, tv, to, tft, tfz, a);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

namespace {
// One thread waits on a barrier nothing arrives at; the bounded wait gives
// up after limit_ns and records the timeout like a real stalled launch.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::fence_mbar_init();
        if (!sm100::mbar_wait(&bar, 0, limit_ns)) atomicAdd(&g_tc_timeouts, 1u);
    }
}
}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

unsigned int take_tc_timeouts() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_timeouts, sizeof(v)) != cudaSuccess) return 0;
    cudaMemcpyToSymbol(g_tc_timeouts, &zero, sizeof(zero));
    return v;
}

}  // namespace kda
