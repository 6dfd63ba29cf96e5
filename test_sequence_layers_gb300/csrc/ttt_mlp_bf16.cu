// ttt_mlp_bf16.cu -- TTT-MLP forward on sm_103a: bf16 operands, fp32
// accumulation, fp32 inner-weight state.
//
// Inner model f(x) = act(x W1 + c1) W2 + c2, act = SiLU or GELU (template ACT; the
// derivation below is written for SiLU and holds for any act with act' in place of
// SiLU'), two layers, hidden width m = 4d (
// "Learning to (Learn at Test Time)" walkthrough, section 2.2.1; SiLU and the
// width ratio 4 of the ViT3 article, observation 4).  For one mini-batch
// (chunk of <= 16 tokens here) with start weights, the per-token gradients of
// 1/2 ||f(k_s) - v_s||^2 and their cumulative effect on the queries are, with
// h_s = k_s W1 + c1, a_s = SiLU(h_s), e_s = a_s W2 + c2 - v_s,
// delta_s = (e_s W2^T) .* SiLU'(h_s), Et = diag(eta) E, Dt = diag(eta) Delta:
//     H_q = Q W1 + c1 - (M .* (Q K^T + 1)) Dt          (W1, c1 after the writes s <= t)
//     Z   = SiLU(H_q) W2 + c2 - (M .* (SiLU(H_q) A_k^T + 1)) Et
//     W1 -= K^T Dt,  c1 -= 1^T Dt,  W2 -= A_k^T Et,  c2 -= 1^T Et
// where M is the lower-triangular mask with diagonal (causal) or all ones
// (queries read the block-end weights); the "+1" carries the bias writes.
// This is the dual (matrix) form of the mini-batch rule (walkthrough section
// 1.2.2) applied to the two-layer model; SiLU'(h) = sigma(h) (1 + h (1 - sigma(h))).
//
// Work split (one CTA per (batch, head) chain, 16 warps at d = 64):
//  * warp w owns hidden units [16w, 16w+16): W1^T rows (fp32, registers), W2^T
//    columns (fp32, shared memory), c1 entries; it computes H_k, A_k, delta and
//    both weight updates for them, and H_q / A_q;
//  * "column warps" c < d/8 own output columns [8c, 8c+8) of E, of the query
//    product P = A_q W2 and of Z: those contract over all hidden units, read
//    from shared memory (A_k, A_q and a bf16 copy of W2), so no cross-warp
//    reduction is needed;
//  * two "score warps" form S2 = A_q A_k^T.
// Four CTA barriers separate the phases of a chunk.  Warp 0 issues the TMA loads
// of the Q/K/V tiles a few chunks ahead (3-stage ring, mbarrier completion).
// All products are warp-level mma.sync m16n8k16 (bf16 in, fp32 accumulate).
#include <cuda.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"
#include "ttt_jobs.cuh"

namespace ttt {

template <int D>
struct MlpCfg {
    static constexpr int M = 4 * D;               // hidden width
    static constexpr int NW = M / 16;             // warps (16 hidden units each)
    static constexpr int THREADS = NW * 32;
    static constexpr int NCOL = D / 8;            // column warps (8 output columns each)
    static constexpr int NK = D / 16;             // 16-wide k-tiles along d
    static constexpr int NKM = M / 16;            // 16-wide k-tiles along m
    static constexpr int NS = 3;                  // token tile stages
    static constexpr int RB = 2 * D;              // bytes per tile row (D <= 64)
    static constexpr int TILE = 16 * D * 2;
    static constexpr int TILE_A = ((TILE + 1023) / 1024) * 1024;
    static constexpr int STAGE = ((3 * TILE_A + 64 + 1023) / 1024) * 1024;  // Q, K, V, eta
    static constexpr int W2R = 2 * D + 16;        // bf16 W2 row stride [hidden][d]
    static constexpr int AR = 2 * M + 16;         // bf16 A_k / A_q row stride [tok][hidden]
    static constexpr int ER = 2 * D + 16;         // bf16 E / -Et row stride [tok][d]
    static constexpr int SR = 48;                 // bf16 16x16 row stride
    static constexpr int W2F_OFF = NS * STAGE;    // fp32 W2^T slices, fragment order
    static constexpr int W2B_OFF = W2F_OFF + M * D * 4;   // bf16 W2 [M][W2R]
    static constexpr int AK_OFF = W2B_OFF + M * W2R;      // bf16 A_k [16][AR]
    static constexpr int AQ_OFF = AK_OFF + 16 * AR;       // bf16 A_q [16][AR]
    static constexpr int EB_OFF = AQ_OFF + 16 * AR;       // bf16 E
    static constexpr int NEB_OFF = EB_OFF + 16 * ER;      // bf16 -Et
    static constexpr int SP_OFF = NEB_OFF + 16 * ER;      // bf16 M .* (Q K^T + 1)
    static constexpr int S2_OFF = SP_OFF + 16 * SR;       // bf16 M .* (A_q A_k^T + 1)
    static constexpr int BAR_OFF = ((S2_OFF + 16 * SR + 15) / 16) * 16;
    static constexpr int SMEM = BAR_OFF + NS * 8 + 16 + 1024;
    // causal mini-batches of several chunks: bf16 copies of the current weights
    // (the queries' weights) next to the block-start copies the residuals read
    static constexpr int W2C_OFF = ((BAR_OFF + NS * 8 + 16 + 127) / 128) * 128;  // bf16 W2 [M][W2R]
    static constexpr int W1C_OFF = W2C_OFF + M * W2R;             // bf16 W1^T [M][W2R]
    static constexpr int SMEM_MULTI = W1C_OFF + M * W2R + 1024;
    // otherwise: the W2C region is the second of two bf16 W2 buffers (the copy of the
    // next mini-batch's start weights is written while the current one is read)
    static constexpr int SMEM_DBL = W2C_OFF + M * W2R + 1024;
    static constexpr uint32_t SWM = RB == 128 ? 7u : (RB == 64 ? 3u : 1u);
};

// Byte offset of element (r, c) of a 16 x D bf16 tile written by TMA with the
// swizzle matching the row length (16-byte chunk index XOR the 128-byte line).
template <int D>
__device__ __forceinline__ uint32_t mtoff(int r, int c)
{
    uint32_t a = static_cast<uint32_t>(r * MlpCfg<D>::RB + c * 2);
    return a ^ (((a >> 7) & MlpCfg<D>::SWM) << 4);
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void stsm_x4_t(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3)
{
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

// logistic function as (1 + tanh(h / 2)) / 2 with the hardware tanh approximation: one
// special-function op per value instead of an exponential and a reciprocal
__device__ __forceinline__ float sigmoid_f(float h)
{
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * h));
    return fmaf(0.5f, t, 0.5f);
}

// Inner activation: ACT 0 = SiLU(h) = h sigma(h) (ViT3 article, observation 4),
// ACT 1 = GELU(h) = h Phi(h), Phi the standard normal CDF (the walkthrough's TTT-MLP,
// section 2.2.1; norm_cdf: erf by Abramowitz & Stegun 7.1.26).  act() gives the value, act_d() the value
// and the derivative (SiLU' = sigma (1 + h (1 - sigma)), GELU' = Phi + h phi).
template <int ACT>
__device__ __forceinline__ float act(float h)
{
    if constexpr (ACT == 0) return h * sigmoid_f(h);
    else {
        float e;
        return h * norm_cdf(h, e);
    }
}

template <int ACT>
__device__ __forceinline__ void act_d(float h, float &a, float &ad)
{
    if constexpr (ACT == 0) {
        const float sg = sigmoid_f(h);
        a = h * sg;
        ad = sg * (1.f + h * (1.f - sg));
    } else {
        float e;
        const float Phi = norm_cdf(h, e);
        a = h * Phi;
        ad = fmaf(h * 0.39894228040143268f, e, Phi);
    }
}

struct MlpParams {
    int H, T, b, causal, per_batch;
    const float *eta;
    float eta_scalar;
    const float *W1, *c1, *W2, *c2;
    __nv_bfloat16 *z;
    float *W1o, *c1o, *W2o, *c2o;
    int *status;
};

// The eight-warp kernel with the inner norm + residual: [H][d] scale and shift, and
// the queries (the residual of z, read from global memory).
struct MlpLnParams : MlpParams {
    const float *ln_gamma, *ln_beta;
    float ln_eps;
    const __nv_bfloat16 *q;
};

// MULTI: causal with mini-batches longer than one 16-token chunk, so the chunk's
// queries read weights that already include the earlier chunks' writes while its
// residuals are taken at the mini-batch's start weights.
template <int D, bool MULTI, int ACT>
__global__ void __launch_bounds__(MlpCfg<D>::THREADS, 1)
    ttt_mlp_bf16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const MlpParams p)
{
    using C = MlpCfg<D>;
    constexpr int M = C::M, NK = C::NK, NKM = C::NKM, NJ = D / 8, NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x, T = p.T;
    const int g = lane >> 2, t4 = lane & 3;
    // ldmatrix / stmatrix lane address patterns (row within a 16-row tile, column offset)
    //  A: blocks (rows 0-7, c), (rows 8-15, c), (rows 0-7, c+8), (rows 8-15, c+8)
    //  B: blocks (rows 0-7, c), (rows 0-7, c+8), (rows 8-15, c), (rows 8-15, c+8)
    const int rowA = (lane & 7) + 8 * ((lane >> 3) & 1), colA = 8 * (lane >> 4);
    const int rowB = (lane & 7) + 8 * (lane >> 4), colB = 8 * ((lane >> 3) & 1);
    const bool has_eta = p.eta != nullptr;
    const uint32_t bar_full = base + C::BAR_OFF;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + C::BAR_OFF + NS * 8);
    const uint32_t AK = base + C::AK_OFF, AQ = base + C::AQ_OFF;
    int w2cur = 0;  // which bf16 W2 buffer holds the current mini-batch's start weights
    const uint32_t EB = base + C::EB_OFF, NEB = base + C::NEB_OFF;
    const uint32_t SP = base + C::SP_OFF, S2P = base + C::S2_OFF;
    const uint32_t W2C = base + C::W2C_OFF, W1C = base + C::W1C_OFF;  // used when MULTI

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bar_full + 8 * s, 1 + (has_eta ? 32 : 0));
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ---------------------------------------------------------- initial state
    const int w = warp, h0 = 16 * w;
    const bool colw = w < C::NCOL;  // owns output columns [8w, 8w+8)
    const int c0 = 8 * w;
    const size_t ps = p.per_batch ? (size_t)bh : (size_t)(bh % p.H);
    const float *W1g = p.W1 + ps * D * M, *c1g = p.c1 + ps * M;
    const float *W2g = p.W2 + ps * M * D, *c2g = p.c2 + ps * D;
    // W1^T rows h0.. of this warp: w1[j][0..1] = W1[8j+2t4 .. +1][h0+g], [2..3] = column h0+g+8
    float w1[NJ][4];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int r = 8 * j + 2 * t4;
        w1[j][0] = W1g[(size_t)r * M + h0 + g];
        w1[j][1] = W1g[(size_t)(r + 1) * M + h0 + g];
        w1[j][2] = W1g[(size_t)r * M + h0 + g + 8];
        w1[j][3] = W1g[(size_t)(r + 1) * M + h0 + g + 8];
    }
    float c1r[2][2], c1s[2][2];  // c1 of hidden h0 + 8nt + 2t4 + i (current, block start)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 2; ++i) c1r[nt][i] = c1s[nt][i] = c1g[h0 + 8 * nt + 2 * t4 + i];
    // W2^T columns h0.. of this warp, fp32 in shared memory in fragment order:
    // tile (mt, nt) holds W2[h0+8nt+2t4 .. +1][16mt+g] and [..][16mt+g+8]
    auto w2f = [&](int mt, int nt) -> uint32_t {
        return base + C::W2F_OFF + (uint32_t)(((w * NK + mt) * 2 + nt) * 32 + lane) * 16;
    };
#pragma unroll
    for (int mt = 0; mt < NK; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int hr = h0 + 8 * nt + 2 * t4, dc = 16 * mt + g;
            const float x = W2g[(size_t)hr * D + dc], y = W2g[(size_t)(hr + 1) * D + dc];
            const float zz = W2g[(size_t)hr * D + dc + 8], ww = W2g[(size_t)(hr + 1) * D + dc + 8];
            asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(w2f(mt, nt)), "f"(x), "f"(y),
                         "f"(zz), "f"(ww)
                         : "memory");
        }
    float c2r[2] = {0.f, 0.f}, c2s[2] = {0.f, 0.f};  // c2 of columns c0 + 2t4 + i (column warps)
    if (colw) {
        c2r[0] = c2s[0] = c2g[c0 + 2 * t4];
        c2r[1] = c2s[1] = c2g[c0 + 2 * t4 + 1];
    }
    uint32_t w1b[2 * NJ];  // bf16 W1 as B operand: word 4kk + nt (tile 2kk), 4kk + 2 + nt (tile 2kk+1)

    // ------------------------------------------------ token tiles (warp 0 issues)
    JobIter itp(T, p.b, p.causal);
    int issued = 0;
    auto issue_next = [&]() {
        if (!itp.valid()) return;
        const Job J = itp.get();
        const int s = issued % NS;
        const uint32_t st = base + s * C::STAGE, full = bar_full + 8 * s;
        if (has_eta) {
            if (J.kind != kOut && lane < J.c)
                cp_async_4(st + 3 * C::TILE_A + 4 * lane, p.eta + (size_t)bh * T + J.t0 + lane);
            cp_async_arrive_noinc(full);
        }
        if (lane == 0) {
            const bool lq = J.kind != kUpd, lkv = J.kind != kOut;
            mbar_arrive_expect_tx(full, (uint32_t)((lq ? 1 : 0) + (lkv ? 2 : 0)) * C::TILE);
            if (lq) tma_load_3d(st, &tq, full, 0, J.t0, bh);
            if (lkv) {
                tma_load_3d(st + C::TILE_A, &tk, full, 0, J.t0, bh);
                tma_load_3d(st + 2 * C::TILE_A, &tv, full, 0, J.t0, bh);
            }
        }
        __syncwarp();
        itp.next();
        ++issued;
    };
    if (warp == 0)
        for (int i = 0; i < NS - 1; ++i) issue_next();

    // ---------------------------------------------------------------- chunks
    JobIter it(T, p.b, p.causal);
    for (int jb = 0; it.valid(); it.next(), ++jb) {
        const Job J = it.get();
        if (warp == 0) issue_next();  // into the stage the previous chunk released
        const int s = jb % NS;
        const uint32_t st = base + s * C::STAGE;
        const uint32_t tQ = st, tK = st + C::TILE_A, tV = st + 2 * C::TILE_A;
        const float *eta_s = reinterpret_cast<const float *>(gbase + s * C::STAGE + 3 * C::TILE_A);
        const bool upd = J.kind != kOut, out = J.kind != kUpd, both = J.kind == kBoth;
        auto eta_of = [&](int tok) -> float { return has_eta ? eta_s[tok] : p.eta_scalar; };
        // bf16 W2 [hidden][d] at the start of this mini-batch (the residuals read it;
        // so do the queries unless MULTI), and the buffer for the next one
        const uint32_t W2B = base + (w2cur ? C::W2C_OFF : C::W2B_OFF);
        const uint32_t W2N = base + (w2cur ? C::W2B_OFF : C::W2C_OFF);
        const uint32_t W2Q = MULTI ? W2C : W2B;  // W2 the queries read

        // phase 0: bf16 copies of the weights this pass reads (start of a
        // mini-batch for the residuals; block-end weights for a query pass)
        if (J.first) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int o = 4 * (j >> 1) + 2 * (j & 1);
                w1b[o] = pack_bf16(w1[j][0], w1[j][1]);
                w1b[o + 1] = pack_bf16(w1[j][2], w1[j][3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                c1s[nt][0] = c1r[nt][0];
                c1s[nt][1] = c1r[nt][1];
            }
            c2s[0] = c2r[0];
            c2s[1] = c2r[1];
        }
        // W2 as bf16 [hidden][d] (transposed stores of the W2^T fragments).  Without
        // MULTI only the first chunk converts: each mini-batch's last update writes
        // the next start weights straight from its registers.
        if (MULTI ? J.first : jb == 0) {
#pragma unroll
            for (int mt = 0; mt < NK; ++mt) {
                const uint4 x0 = lds128(w2f(mt, 0)), x1 = lds128(w2f(mt, 1));
                const int blk = lane >> 3, rr = lane & 7;
                const uint32_t addr = W2B + (uint32_t)(h0 + 8 * (blk >> 1) + rr) * C::W2R +
                                      (uint32_t)(16 * mt + 8 * (blk & 1)) * 2;
                stsm_x4_t(addr, pack_bf16(__uint_as_float(x0.x), __uint_as_float(x0.y)),
                          pack_bf16(__uint_as_float(x0.z), __uint_as_float(x0.w)),
                          pack_bf16(__uint_as_float(x1.x), __uint_as_float(x1.y)),
                          pack_bf16(__uint_as_float(x1.z), __uint_as_float(x1.w)));
            }
        }
        if constexpr (MULTI) {
            // current weights for this chunk's queries: W2 [hidden][d] and W1^T
            // [hidden][d_in] as bf16 (this warp's 16 hidden rows of each)
#pragma unroll
            for (int mt = 0; mt < NK; ++mt) {
                const uint4 x0 = lds128(w2f(mt, 0)), x1 = lds128(w2f(mt, 1));
                const int blk = lane >> 3, rr = lane & 7;
                const uint32_t addr = W2C + (uint32_t)(h0 + 8 * (blk >> 1) + rr) * C::W2R +
                                      (uint32_t)(16 * mt + 8 * (blk & 1)) * 2;
                stsm_x4_t(addr, pack_bf16(__uint_as_float(x0.x), __uint_as_float(x0.y)),
                          pack_bf16(__uint_as_float(x0.z), __uint_as_float(x0.w)),
                          pack_bf16(__uint_as_float(x1.x), __uint_as_float(x1.y)),
                          pack_bf16(__uint_as_float(x1.z), __uint_as_float(x1.w)));
            }
#pragma unroll
            for (int kk = 0; kk < NK; ++kk)
                stsm_x4(W1C + (uint32_t)(h0 + rowA) * C::W2R + (16 * kk + colA) * 2,
                        pack_bf16(w1[2 * kk][0], w1[2 * kk][1]), pack_bf16(w1[2 * kk][2], w1[2 * kk][3]),
                        pack_bf16(w1[2 * kk + 1][0], w1[2 * kk + 1][1]),
                        pack_bf16(w1[2 * kk + 1][2], w1[2 * kk + 1][3]));
        }
        if (!mbar_wait(bar_full + 8 * s, (jb / NS) & 1, p.status, kSiteConsumerFull)) *abort_flag = 1;

        // phase 1: H_k = K W1 + c1, A_k = SiLU(H_k) -> shared; scores for the queries
        float ak[2][4], sp[2][4];
        uint32_t akp[4] = {0, 0, 0, 0};
        if (upd) {
            float hk[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(tK + mtoff<D>(rowA, 16 * kk + colA), a0, a1, a2, a3);
                mma_bf16(hk[0], a0, a1, a2, a3, w1b[4 * kk], w1b[4 * kk + 2]);
                mma_bf16(hk[1], a0, a1, a2, a3, w1b[4 * kk + 1], w1b[4 * kk + 3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    act_d<ACT>(hk[nt][i] + c1s[nt][i & 1], ak[nt][i], sp[nt][i]);
                }
            akp[0] = pack_bf16(ak[0][0], ak[0][1]);  // (tok 0-7, hidden 0-7)
            akp[1] = pack_bf16(ak[0][2], ak[0][3]);  // (tok 8-15, hidden 0-7)
            akp[2] = pack_bf16(ak[1][0], ak[1][1]);  // (tok 0-7, hidden 8-15)
            akp[3] = pack_bf16(ak[1][2], ak[1][3]);  // (tok 8-15, hidden 8-15)
            stsm_x4(AK + rowA * C::AR + (h0 + colA) * 2, akp[0], akp[1], akp[2], akp[3]);
        }
        if (both && w == C::NW - 1) {
            // S' = M .* (Q K^T + 1)
            float sc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint32_t a0, a1, a2, a3, b00, b01, b10, b11;
                ldsm_x4(tQ + mtoff<D>(rowA, 16 * kk + colA), a0, a1, a2, a3);
                ldsm_x4(tK + mtoff<D>(rowB, 16 * kk + colB), b00, b01, b10, b11);
                mma_bf16(sc[0], a0, a1, a2, a3, b00, b01);
                mma_bf16(sc[1], a0, a1, a2, a3, b10, b11);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tq_ = g + 8 * (i >> 1), ss = 8 * nt + 2 * t4 + (i & 1);
                    const bool keep = ss < J.c && (!p.causal || ss <= tq_);
                    sc[nt][i] = keep ? sc[nt][i] + 1.f : 0.f;
                }
            stsm_x4(SP + rowA * C::SR + colA * 2, pack_bf16(sc[0][0], sc[0][1]),
                    pack_bf16(sc[0][2], sc[0][3]), pack_bf16(sc[1][0], sc[1][1]),
                    pack_bf16(sc[1][2], sc[1][3]));
        }
        __syncthreads();  // B1: A_k, S', bf16 W2 visible
        if (*abort_flag) break;

        // phase 2: E = A_k W2 + c2 - V on this column warp's 8 columns; -Et
        float cs2[2] = {0.f, 0.f};  // column sums of -Et (c2 write of this chunk)
        if (upd && colw) {
            float e[2][4] = {};
#pragma unroll
            for (int kp = 0; kp < NKM / 2; ++kp) {
                uint32_t b0a, b1a, b0b, b1b, a0, a1, a2, a3, a4, a5, a6, a7;
                ldsm_x4_t(W2B + (uint32_t)(32 * kp + lane) * C::W2R + c0 * 2, b0a, b1a, b0b, b1b);
                ldsm_x4(AK + rowA * C::AR + (32 * kp + colA) * 2, a0, a1, a2, a3);
                ldsm_x4(AK + rowA * C::AR + (32 * kp + 16 + colA) * 2, a4, a5, a6, a7);
                mma_bf16(e[0], a0, a1, a2, a3, b0a, b1a);
                mma_bf16(e[1], a4, a5, a6, a7, b0b, b1b);
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {  // token rows g, g + 8
                const int tok = g + 8 * r;
                const uint32_t vw = *reinterpret_cast<const uint32_t *>(gbase + (tV - base) +
                                                                        mtoff<D>(tok, c0 + 2 * t4));
                const float ex = e[0][2 * r] + e[1][2 * r] + c2s[0] - bf16_lo(vw);
                const float ey = e[0][2 * r + 1] + e[1][2 * r + 1] + c2s[1] - bf16_hi(vw);
                const bool ok = tok < J.c;
                const float et = -eta_of(tok);
                const float nx = ok ? et * ex : 0.f, ny = ok ? et * ey : 0.f;
                cs2[0] += nx;
                cs2[1] += ny;
                *reinterpret_cast<uint32_t *>(gbase + C::EB_OFF + tok * C::ER + (c0 + 2 * t4) * 2) =
                    pack_bf16(ex, ey);
                *reinterpret_cast<uint32_t *>(gbase + C::NEB_OFF + tok * C::ER + (c0 + 2 * t4) * 2) =
                    pack_bf16(nx, ny);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                cs2[i] += __shfl_xor_sync(0xffffffffu, cs2[i], 4);
                cs2[i] += __shfl_xor_sync(0xffffffffu, cs2[i], 8);
                cs2[i] += __shfl_xor_sync(0xffffffffu, cs2[i], 16);
            }
        }
        __syncthreads();  // B2: E, -Et visible

        // phase 3: delta, weight updates, query pre-activations
        uint32_t d00 = 0, d01 = 0, d10 = 0, d11 = 0;  // -Dt^T blocks (hidden x tok)
        float cs1[2][2] = {};                         // column sums of -Dt (c1 write)
        if (upd) {
            float dl[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                ldsm_x4(EB + rowA * C::ER + (16 * kk + colA) * 2, a0, a1, a2, a3);
                ldsm_x4(W2B + (uint32_t)(h0 + rowB) * C::W2R + (16 * kk + colB) * 2, b0, b1, b2, b3);
                mma_bf16(dl[0], a0, a1, a2, a3, b0, b1);
                mma_bf16(dl[1], a0, a1, a2, a3, b2, b3);
            }
            float nd[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tok = g + 8 * (i >> 1);
                    nd[nt][i] = tok < J.c ? -eta_of(tok) * dl[nt][i] * sp[nt][i] : 0.f;
                    cs1[nt][i & 1] += nd[nt][i];
                }
            d00 = movmatrix_t(pack_bf16(nd[0][0], nd[0][1]));  // (hidden 0-7, tok 0-7)
            d01 = movmatrix_t(pack_bf16(nd[1][0], nd[1][1]));  // (hidden 8-15, tok 0-7)
            d10 = movmatrix_t(pack_bf16(nd[0][2], nd[0][3]));  // (hidden 0-7, tok 8-15)
            d11 = movmatrix_t(pack_bf16(nd[1][2], nd[1][3]));  // (hidden 8-15, tok 8-15)
            // W1^T += (-Dt^T) K
#pragma unroll
            for (int j2 = 0; j2 < NK; ++j2) {
                uint32_t k0, k1, k2, k3;
                ldsm_x4_t(tK + mtoff<D>(rowA, 16 * j2 + colA), k0, k1, k2, k3);
                mma_bf16(w1[2 * j2], d00, d01, d10, d11, k0, k1);
                mma_bf16(w1[2 * j2 + 1], d00, d01, d10, d11, k2, k3);
            }
            // W2^T += (-Et^T) A_k (fp32 slices in shared memory); the last update of a
            // mini-batch also writes the bf16 copy of the next start weights
            const uint32_t bt00 = movmatrix_t(akp[0]), bt01 = movmatrix_t(akp[1]);
            const uint32_t bt10 = movmatrix_t(akp[2]), bt11 = movmatrix_t(akp[3]);
            const bool put_next = !MULTI && J.last_upd;
#pragma unroll
            for (int mt = 0; mt < NK; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(NEB + rowB * C::ER + (16 * mt + colB) * 2, a0, a1, a2, a3);
                float x0[4], x1[4];
                const uint4 u0 = lds128(w2f(mt, 0)), u1 = lds128(w2f(mt, 1));
                x0[0] = __uint_as_float(u0.x); x0[1] = __uint_as_float(u0.y);
                x0[2] = __uint_as_float(u0.z); x0[3] = __uint_as_float(u0.w);
                x1[0] = __uint_as_float(u1.x); x1[1] = __uint_as_float(u1.y);
                x1[2] = __uint_as_float(u1.z); x1[3] = __uint_as_float(u1.w);
                mma_bf16(x0, a0, a1, a2, a3, bt00, bt01);
                mma_bf16(x1, a0, a1, a2, a3, bt10, bt11);
                asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(w2f(mt, 0)), "f"(x0[0]),
                             "f"(x0[1]), "f"(x0[2]), "f"(x0[3])
                             : "memory");
                asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(w2f(mt, 1)), "f"(x1[0]),
                             "f"(x1[1]), "f"(x1[2]), "f"(x1[3])
                             : "memory");
                if (put_next) {
                    const int blk = lane >> 3, rr = lane & 7;
                    const uint32_t addr = W2N + (uint32_t)(h0 + 8 * (blk >> 1) + rr) * C::W2R +
                                          (uint32_t)(16 * mt + 8 * (blk & 1)) * 2;
                    stsm_x4_t(addr, pack_bf16(x0[0], x0[1]), pack_bf16(x0[2], x0[3]), pack_bf16(x1[0], x1[1]),
                              pack_bf16(x1[2], x1[3]));
                }
            }
        }
        if (out) {
            // H_q = Q W1 + c1 + S' (-Dt); A_q = SiLU(H_q) -> shared
            float hq[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(tQ + mtoff<D>(rowA, 16 * kk + colA), a0, a1, a2, a3);
                if constexpr (MULTI) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(W1C + (uint32_t)(h0 + rowB) * C::W2R + (16 * kk + colB) * 2, b0, b1, b2, b3);
                    mma_bf16(hq[0], a0, a1, a2, a3, b0, b1);
                    mma_bf16(hq[1], a0, a1, a2, a3, b2, b3);
                } else {
                    mma_bf16(hq[0], a0, a1, a2, a3, w1b[4 * kk], w1b[4 * kk + 2]);
                    mma_bf16(hq[1], a0, a1, a2, a3, w1b[4 * kk + 1], w1b[4 * kk + 3]);
                }
            }
            if (both) {
                uint32_t s0, s1, s2, s3;
                ldsm_x4(SP + rowA * C::SR + colA * 2, s0, s1, s2, s3);
                mma_bf16(hq[0], s0, s1, s2, s3, d00, d10);
                mma_bf16(hq[1], s0, s1, s2, s3, d01, d11);
            }
            float aq[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    aq[nt][i] = act<ACT>(hq[nt][i] + c1r[nt][i & 1]);
                }
            stsm_x4(AQ + rowA * C::AR + (h0 + colA) * 2, pack_bf16(aq[0][0], aq[0][1]),
                    pack_bf16(aq[0][2], aq[0][3]), pack_bf16(aq[1][0], aq[1][1]),
                    pack_bf16(aq[1][2], aq[1][3]));
        }
        if (upd) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    float v = cs1[nt][i];
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    c1r[nt][i] += v;
                }
        }
        __syncthreads();  // B3: A_q visible; the stage's tiles are no longer read

        // phase 4: P = A_q W2, S2' = M .* (A_q A_k^T + 1), Z = P + c2 + S2' (-Et)
        if (out) {
            float pz[2][4] = {};
            if (colw) {
#pragma unroll
                for (int kp = 0; kp < NKM / 2; ++kp) {
                    uint32_t b0a, b1a, b0b, b1b, a0, a1, a2, a3, a4, a5, a6, a7;
                    ldsm_x4_t(W2Q + (uint32_t)(32 * kp + lane) * C::W2R + c0 * 2, b0a, b1a, b0b, b1b);
                    ldsm_x4(AQ + rowA * C::AR + (32 * kp + colA) * 2, a0, a1, a2, a3);
                    ldsm_x4(AQ + rowA * C::AR + (32 * kp + 16 + colA) * 2, a4, a5, a6, a7);
                    mma_bf16(pz[0], a0, a1, a2, a3, b0a, b1a);
                    mma_bf16(pz[1], a4, a5, a6, a7, b0b, b1b);
                }
            } else if (both && w < C::NCOL + 2) {
                const int u = w - C::NCOL;  // key tokens 8u .. 8u+7
                float s2[2][4] = {};
#pragma unroll
                for (int kp = 0; kp < NKM / 2; ++kp) {
                    uint32_t b0, b1, b2, b3, a0, a1, a2, a3, a4, a5, a6, a7;
                    ldsm_x4(AK + (uint32_t)(8 * u + (lane & 7)) * C::AR + (32 * kp + 8 * (lane >> 3)) * 2,
                            b0, b1, b2, b3);
                    ldsm_x4(AQ + rowA * C::AR + (32 * kp + colA) * 2, a0, a1, a2, a3);
                    ldsm_x4(AQ + rowA * C::AR + (32 * kp + 16 + colA) * 2, a4, a5, a6, a7);
                    mma_bf16(s2[0], a0, a1, a2, a3, b0, b1);
                    mma_bf16(s2[1], a4, a5, a6, a7, b2, b3);
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {  // query rows g, g + 8
                    const int tq_ = g + 8 * r;
                    float v[2];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int ss = 8 * u + 2 * t4 + i;
                        const bool keep = ss < J.c && (!p.causal || ss <= tq_);
                        v[i] = keep ? s2[0][2 * r + i] + s2[1][2 * r + i] + 1.f : 0.f;
                    }
                    *reinterpret_cast<uint32_t *>(gbase + C::S2_OFF + tq_ * C::SR + (8 * u + 2 * t4) * 2) =
                        pack_bf16(v[0], v[1]);
                }
            }
            __syncthreads();  // B4: S2' visible
            if (colw) {
                float zz[4] = {pz[0][0] + pz[1][0], pz[0][1] + pz[1][1], pz[0][2] + pz[1][2],
                               pz[0][3] + pz[1][3]};
                if (both) {
                    uint32_t s0, s1, s2, s3, b0, b1, b2, b3;
                    ldsm_x4(S2P + rowA * C::SR + colA * 2, s0, s1, s2, s3);
                    ldsm_x4_t(NEB + (uint32_t)(lane & 15) * C::ER + c0 * 2, b0, b1, b2, b3);
                    mma_bf16(zz, s0, s1, s2, s3, b0, b1);
                }
                __nv_bfloat16 *zb = p.z + ((size_t)bh * T + J.t0) * D + c0 + 2 * t4;
                if (g < J.c)
                    *reinterpret_cast<uint32_t *>(zb + (size_t)g * D) =
                        pack_bf16(zz[0] + c2r[0], zz[1] + c2r[1]);
                if (g + 8 < J.c)
                    *reinterpret_cast<uint32_t *>(zb + (size_t)(g + 8) * D) =
                        pack_bf16(zz[2] + c2r[0], zz[3] + c2r[1]);
            }
        }
        if (upd && colw) {
            c2r[0] += cs2[0];
            c2r[1] += cs2[1];
        }
        if (!MULTI && J.last_upd) w2cur ^= 1;
    }

    // ------------------------------------------------------------ final state
    if (p.W1o) {
        float *o = p.W1o + (size_t)bh * D * M;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int r = 8 * j + 2 * t4;
            o[(size_t)r * M + h0 + g] = w1[j][0];
            o[(size_t)(r + 1) * M + h0 + g] = w1[j][1];
            o[(size_t)r * M + h0 + g + 8] = w1[j][2];
            o[(size_t)(r + 1) * M + h0 + g + 8] = w1[j][3];
        }
    }
    if (p.c1o && g == 0) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 2; ++i) p.c1o[(size_t)bh * M + h0 + 8 * nt + 2 * t4 + i] = c1r[nt][i];
    }
    if (p.W2o) {
        float *o = p.W2o + (size_t)bh * M * D;
#pragma unroll
        for (int mt = 0; mt < NK; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const uint4 u = lds128(w2f(mt, nt));
                const int hr = h0 + 8 * nt + 2 * t4, dc = 16 * mt + g;
                o[(size_t)hr * D + dc] = __uint_as_float(u.x);
                o[(size_t)(hr + 1) * D + dc] = __uint_as_float(u.y);
                o[(size_t)hr * D + dc + 8] = __uint_as_float(u.z);
                o[(size_t)(hr + 1) * D + dc + 8] = __uint_as_float(u.w);
            }
    }
    if (p.c2o && colw && g == 0) {
        p.c2o[(size_t)bh * D + c0 + 2 * t4] = c2r[0];
        p.c2o[(size_t)bh * D + c0 + 2 * t4 + 1] = c2r[1];
    }
    // make sure no copy is still landing in shared memory when the CTA ends
    if (warp == 0)
        for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
            if (!mbar_wait(bar_full + 8 * (j % NS), (j / NS) & 1, p.status, kSiteDrain)) break;
}

template <int D>
static int launch_mlp_t(const MlpArgs &a, const CUtensorMap *maps)
{
    using C = MlpCfg<D>;
    const bool multi = a.causal && a.b > 16;
    auto kern = multi ? (a.act ? ttt_mlp_bf16_kernel<D, true, 1> : ttt_mlp_bf16_kernel<D, true, 0>)
                      : (a.act ? ttt_mlp_bf16_kernel<D, false, 1> : ttt_mlp_bf16_kernel<D, false, 0>);
    const int smem = multi ? C::SMEM_MULTI : C::SMEM_DBL;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return -4;
    MlpParams p;
    p.H = a.H;
    p.T = a.T;
    p.b = a.b;
    p.causal = a.causal;
    p.per_batch = a.per_batch;
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W1 = a.W1;
    p.c1 = a.c1;
    p.W2 = a.W2;
    p.c2 = a.c2;
    p.z = static_cast<__nv_bfloat16 *>(a.z);
    p.W1o = a.W1o;
    p.c1o = a.c1o;
    p.W2o = a.W2o;
    p.c2o = a.c2o;
    p.status = a.status;
    kern<<<a.B * a.H, C::THREADS, smem, a.stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// ---------------------------------------------------------------------------
// Eight-warp kernel for d = 64 (m = 256) and mini-batches of at most 16 tokens
// (one chunk per mini-batch).  Same algebra as above; the work split differs:
//  * warp w owns hidden units [32w, 32w + 32) as two groups of 16 and keeps the
//    rows of W1^T and W2 for them in registers as fp32 mma accumulators (no
//    shared-memory read-modify-write of W2), updating both with mma.sync;
//  * every warp is also the column warp of output columns [8w, 8w + 8) for the
//    products that contract over all hidden units (E = A_k W2, P = A_q W2);
//  * A_q A_k^T is formed as eight per-warp partial sums over each warp's own
//    hidden units, straight from registers;
//  * warp 0 also issues the TMA loads a few chunks ahead into a four-stage ring
//    (eight warps: two per SM sub-partition, so each may hold up to 255 registers);
//  * the bf16 copy of W2 that the contractions read is double-buffered: each
//    update writes the next mini-batch's copy from registers while the current
//    copy is still read.
struct W8Cfg {
    static constexpr int D = 64, M = 256, NW = 8, THREADS = NW * 32;
    static constexpr int NK = D / 16, NKM = M / 16, NJ = D / 8, NS = 4;
    static constexpr int TILE = 16 * D * 2;                     // one 16-token tile
    static constexpr int STAGE = ((3 * TILE + 64 + 1023) / 1024) * 1024;  // Q, K, V, eta
    static constexpr int W2R = 2 * D + 16, AR = 2 * M + 16, ER = 2 * D + 16;
    static constexpr int W2B_OFF = NS * STAGE;                  // two bf16 W2 [M][W2R]
    static constexpr int AK_OFF = W2B_OFF + 2 * M * W2R;        // bf16 A_k [16][AR]
    static constexpr int AQ_OFF = AK_OFF + 16 * AR;             // bf16 A_q [16][AR]
    static constexpr int EB_OFF = AQ_OFF + 16 * AR;             // bf16 E [2][16][ER] (by chunk parity)
    static constexpr int NEB_OFF = EB_OFF + 2 * 16 * ER;        // bf16 -Et [2][16][ER]
    static constexpr int S2R = 20;                              // fp32 row stride of a partial (bank spread)
    static constexpr int SP_OFF = NEB_OFF + 2 * 16 * ER;        // bf16 S' = M .* (Q K^T + 1) [16][48 B]
    static constexpr int S2P_OFF = SP_OFF + 16 * 48;            // bf16 S2' = M .* (A_q A_k^T + 1) [16][48 B]
    static constexpr int S2F_OFF = S2P_OFF + 16 * 48;           // fp32 [NW][16][S2R] partial A_q A_k^T
    static constexpr int C2S_OFF = S2F_OFF + NW * 16 * S2R * 4; // fp32 [2][D] c2 at a chunk's start
    static constexpr int BAR_OFF = C2S_OFF + 2 * D * 4;         // full[NS], abort flag
    static constexpr int SMEM = BAR_OFF + NS * 8 + 16 + 1024;
};
static_assert(MlpCfg<64>::RB == 128, "tile rows of 128 bytes");
static_assert(W8Cfg::SMEM <= 227 * 1024, "shared memory");


// The inner-norm variant's layout: the plain layout plus the statistics exchange
// (float2 [3][4 warps][16 rows]) after the barriers.
struct W8LnCfg : W8Cfg {
    static constexpr int LNR_OFF = W8Cfg::BAR_OFF + W8Cfg::NS * 8 + 16;
    static constexpr int SMEM = LNR_OFF + 3 * 4 * 16 * 8 + 1024;
};
static_assert(W8LnCfg::SMEM <= 227 * 1024, "shared memory");

// Inner norm of the eight-warp kernel: per-token sums (a, b) over the 64 outputs for
// token rows g and g + 8 -- this warp's 16 columns (quad shuffle), then the four warps of
// its group (float2 buffer red[4 warps][16 rows], named barrier barid of 128 threads).
__device__ __forceinline__ void w8_row_sums(float (&a)[2], float (&b)[2], float2 *red, int wq, int g, int t4,
                                            int barid)
{
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        a[r] += __shfl_xor_sync(0xffffffffu, a[r], 1);
        a[r] += __shfl_xor_sync(0xffffffffu, a[r], 2);
        b[r] += __shfl_xor_sync(0xffffffffu, b[r], 1);
        b[r] += __shfl_xor_sync(0xffffffffu, b[r], 2);
    }
    if (t4 == 0) {
        red[wq * 16 + g] = make_float2(a[0], b[0]);
        red[wq * 16 + g + 8] = make_float2(a[1], b[1]);
    }
    asm volatile("bar.sync %0, 128;" ::"r"(barid) : "memory");
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        a[r] = b[r] = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 x = red[u * 16 + g + 8 * r];
            a[r] += x.x;
            b[r] += x.y;
        }
    }
}

#define W8_LN 0
#define W8_KERNEL ttt_mlp_w8_kernel
#define W8_CFG W8Cfg
#define W8_PARAMS MlpParams
#include "ttt_mlp_w8.cuh"
#undef W8_LN
#undef W8_KERNEL
#undef W8_CFG
#undef W8_PARAMS
#define W8_LN 1
#define W8_KERNEL ttt_mlp_w8_ln_kernel
#define W8_CFG W8LnCfg
#define W8_PARAMS MlpLnParams
#include "ttt_mlp_w8.cuh"
#undef W8_LN
#undef W8_KERNEL
#undef W8_CFG
#undef W8_PARAMS

static int launch_mlp_w8(const MlpArgs &a, const CUtensorMap *maps)
{
    MlpLnParams p;
    p.H = a.H;
    p.T = a.T;
    p.b = a.b;
    p.causal = a.causal;
    p.per_batch = a.per_batch;
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W1 = a.W1;
    p.c1 = a.c1;
    p.W2 = a.W2;
    p.c2 = a.c2;
    p.z = static_cast<__nv_bfloat16 *>(a.z);
    p.W1o = a.W1o;
    p.c1o = a.c1o;
    p.W2o = a.W2o;
    p.c2o = a.c2o;
    p.status = a.status;
    p.ln_gamma = a.ln_gamma;
    p.ln_beta = a.ln_beta;
    p.ln_eps = a.ln_eps;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    if (a.ln_gamma) {
        auto kern = a.act ? ttt_mlp_w8_ln_kernel<1> : ttt_mlp_w8_ln_kernel<0>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, W8LnCfg::SMEM) != cudaSuccess)
            return -4;
        kern<<<a.B * a.H, W8LnCfg::THREADS, W8LnCfg::SMEM, a.stream>>>(maps[0], maps[1], maps[2], p);
    } else {
        auto kern = a.act ? ttt_mlp_w8_kernel<1> : ttt_mlp_w8_kernel<0>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, W8Cfg::SMEM) != cudaSuccess)
            return -4;
        kern<<<a.B * a.H, W8Cfg::THREADS, W8Cfg::SMEM, a.stream>>>(maps[0], maps[1], maps[2], p);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// d in {16, 32, 64} with hidden width m = 4d.
int launch_mlp_bf16(const MlpArgs &a)
{
    if (a.m != 4 * a.d) return -2;
    CUtensorMap maps[3];
    if (!encode_qkv(maps, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 16)) return -4;
    if (a.ln_gamma) {  // inner norm + residual: d = 64, mini-batches <= 16 or one full batch
        if (a.d == 64 && !a.causal && a.b >= a.T) return launch_mlp_fb_tc(a);
        return a.d == 64 && a.b <= 16 ? launch_mlp_w8(a, maps) : -2;
    }
    switch (a.d) {
    case 16: return launch_mlp_t<16>(a, maps);
    case 32: return launch_mlp_t<32>(a, maps);
    case 64:
        if (!a.causal && a.b >= a.T) return launch_mlp_fb_tc(a);  // one full-batch mini-batch (tcgen05)
        return a.b <= 16 ? launch_mlp_w8(a, maps) : launch_mlp_t<64>(a, maps);
    default: return -2;
    }
}

}  // namespace ttt
