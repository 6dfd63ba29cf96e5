// ttt_linear_b16.cu -- TTT-Linear forward specialised to mini-batches of 16
// tokens (the mini-batch size the walkthrough reports for all its experiments,
// "Learning to (Learn at Test Time)", section 1.2.2 / 4.1), bf16 operands, fp32
// accumulation and fp32 weight state, d in {16, 32, 64}.
//
// The algebra is that of ttt_linear_bf16.cu (dual form of one mini-batch:
// E = K W - V, Z = Q W - (mask .* Q K^T) diag(eta) E, W -= K^T diag(eta) E, with W^T
// held as mma.sync accumulators, 16 output columns per warp).  With b = 16 every
// 16-token chunk is exactly one mini-batch.  The same chunks also carry the delta rule
// (b = 1): a forward substitution turns the residuals at the chunk's start weights into
// each token's own (VAR 3 below), after which the chunk is a mini-batch step.  This
// allows a leaner schedule:
//  * tokens arrive in 64-token blocks (one TMA box per tensor per four chunks);
//    the four chunks of a block are unrolled, so every fragment address is a
//    per-lane constant plus a compile-time offset from the block's base;
//  * the compute warps wait for and release a block once, not per chunk;
//  * each warp forms the scores S = Q K^T of its chunk from fragments already in
//    its registers (K's fragments are the B operand of E as well), masks them in
//    registers and uses them directly as the A operand of S (-Et);
//  * each warp prefetches the next chunk's fragments (K, K^T, Q, V, eta) into a
//    second register set while the current chunk's products run;
//  * full 16-token chunks take a path without per-token bounds masks;
//  * Z is stored straight from the accumulator registers.
//
// Every CTA serves one unit: a token range of one (batch, head) chain, in one of
// three roles.  Unsplit launches have one output unit per chain (the whole
// sequence).  The sequence-parallel path (ttt_linear_seqpar.cu) cuts a chain into
// segments of whole 64-token blocks:
//  * output role: the layer's outputs of a segment from its start weights;
//  * chain role: the state chain of the first segment alone (no query side), whose
//    end weights are the second segment's start;
//  * map role: a later segment's affine map.  One mini-batch step is affine in W,
//        W' = W - K^T diag(eta) (K W - V) = (I - K^T diag(eta) K) W + K^T diag(eta) V,
//    so a segment maps its start weights to its end weights as W -> A W + B.  The
//    map role runs the chain on the d x 2d state X = [A | B] from [I | 0], the
//    columns of A seeing labels V = 0: each column of X is updated as a column of
//    W is, so the per-warp code is the state chain with twice as many warps.
#include <cuda.h>

#include <type_traits>

#include "ttt_device.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

template <int D, bool MAP = false>
struct B16Cfg {
    static constexpr int NCW = (MAP ? 2 : 1) * D / 16;  // compute warps, 16 state columns each
    static constexpr int PW = NCW;                   // producer warp
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int NJ = D / 8, NK = D / 16;
    static constexpr int NB = 4;                     // 64-token blocks in flight
    static constexpr int RB = 2 * D;                 // bytes per token row
    static constexpr int BLK = 64 * RB;              // one tensor's 64-token block
    static constexpr int SLOT = ((3 * BLK + 1023) / 1024) * 1024;  // Q, K, V of one block
    static constexpr int ETA_OFF = NB * SLOT;        // 64 fp32 per block
    static constexpr int BAR_OFF = ETA_OFF + NB * 256;
    // full / empty barriers per block slot, then one barrier nothing arrives at (the
    // timeout test of ttt_debug_wait_limit), then the inner-norm partial sums
    static constexpr int RED_OFF = (BAR_OFF + (2 * NB + 1) * 8 + 15) / 16 * 16;  // [3][NCW][16] float2
    // delta rule: each compute warp's coupling matrix of the chunk, [16 s][16 t] fp32
    static constexpr int DA_OFF = RED_OFF + 3 * NCW * 16 * 8;
    static constexpr int SMEM = DA_OFF + NCW * 1024 + 1024;
};

// Offset of element (r, c) inside a 64-token block written by TMA with the swizzle
// of its row length.  For r = 16q + r0 the swizzle key does not depend on q, so
// offsets of a chunk are this per-lane value plus 16 q RB.
template <int D>
__device__ __forceinline__ uint32_t boff(int r, int c)
{
    constexpr uint32_t SWM = 2 * D == 128 ? 7u : (2 * D == 64 ? 3u : 1u);  // swizzle key mask of the row length
    uint32_t a = static_cast<uint32_t>(r * B16Cfg<D>::RB + c * 2);
    return a ^ (((a >> 7) & SWM) << 4);
}

template <int D>
struct Frag {
    uint32_t kB[D / 16][4];  // K as the B operand of E^T = W^T K^T and of S
    uint32_t kT[D / 16][4];  // K as the B operand of the update (transposed load)
    uint32_t qa[D / 16][4];  // Q as the A operand of Z = Q W
    uint32_t vv[2][2];       // V^T in accumulator layout
    float et[2][2];          // eta of tokens 8nt + 2t4 + i of the chunk
    uint32_t kc[2][2];       // inner norm: K^T of this warp's columns in accumulator layout
    uint32_t qz[4];          // inner norm: Q of this warp's columns in the layout of Z
    uint32_t ka[D / 16][4];  // delta rule: K as the A operand of K K^T
};

enum { kRoleOut = 0, kRoleChain = 1, kRoleMap = 2 };

struct B16Params {
    int BH, H, T, causal;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    __nv_bfloat16 *z;
    float *W_out;
    int *status;
    // units: CTA u serves chain u / nseg, segment s = seg0 + u % nseg; segment 0 is
    // tokens [0, len0), segment s >= 1 is [len0 + (s-1) seg_len, len0 + s seg_len)
    // cut at T (len0 and seg_len multiples of 64)
    int len0, seg_len, nseg, seg0, nsplit;  // nsplit: segments per chain in the whole pass
    float *Wst;   // [BH][nsplit-1][d][d] start weights of segments 1 .. nsplit-1
    float *maps;  // [BH][nsplit-2][2][d][d] affine maps A, B of segments 1 .. nsplit-2
    const float *ln_gamma, *ln_beta;  // [H][d] inner norm scale / shift (VAR 2)
    float ln_eps;
    unsigned long long test_stall_ns;  // > 0: the timeout test (first wait on a dead barrier)
};

// Named barrier of the compute warps (the producer warp does not take part).
__device__ __forceinline__ void bar_compute(int nthreads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// The same barrier with an AND vote: true when every compute thread passed true.
__device__ __forceinline__ bool bar_compute_and(int nthreads, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(nthreads)
        : "memory");
    return r != 0;
}

// One unit (chain bh, segment seg) in role ROLE; the CTA has at least the role's
// warps (extra warps leave after the barrier set-up).
// VAR 0: the MSE loss on f(x) = x W.  VAR 1 (DOT): the negative dot-product
// loss, whose residual is -V whatever W is (no product K W on the chain).  VAR 3
// (DELTA, every role): mini-batches of one token, the delta rule, in chunks of
// 16: the residuals at the chunk's start weights R = K W - V become the tokens' own
// residuals through a forward substitution, e_t = r_t - sum_{s<t} (k_t . k_s) eta_s e_s,
// after which the chunk's output and update are those of a 16-token mini-batch.  VAR 2
// (inner norm, output role only): f(x) = x + LN(x W); the per-token layer-norm
// statistics over the d columns, which four warps hold 16 apiece, are summed
// through shared memory with the compute warps' named barrier (forward statistics
// and backward statistics on the chain, the output's statistics beside it), and the
// block-boundary wait becomes a CTA-uniform vote so every warp meets every barrier.
template <int D, int ROLE, int VAR = 0>
__device__ __forceinline__ void b16_unit(const CUtensorMap *tq, const CUtensorMap *tk, const CUtensorMap *tv,
                                         const B16Params &p, const int bh, const int seg)
{
    constexpr bool MAP = ROLE == kRoleMap, QSIDE = ROLE == kRoleOut;
    constexpr bool DOT = VAR == 1, LN = VAR == 2, DELTA = VAR == 3;
    static_assert(!LN || QSIDE, "the inner norm runs in the output role");
    using C = B16Cfg<D, MAP>;
    constexpr int NJ = C::NJ, NK = C::NK, NB = C::NB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tb = seg == 0 ? 0 : p.len0 + (seg - 1) * p.seg_len;               // first token of the unit
    const int T = max(0, min(p.T, seg == 0 ? p.len0 : tb + p.seg_len) - tb);   // tokens of the unit
    const int nblk = (T + 63) >> 6;
    const bool has_eta = p.eta != nullptr;

    const uint32_t blk_full = base + C::BAR_OFF;      // block landed (producer -> warps)
    const uint32_t blk_empty = blk_full + 8 * NB;     // block released (warps -> producer)
    const uint32_t dead = blk_empty + 8 * NB;          // nothing arrives here (timeout test)
    if (threadIdx.x == 0) {
        if (QSIDE) prefetch_tmap(tq);
        prefetch_tmap(tk);
        prefetch_tmap(tv);
        for (int s = 0; s < NB; ++s) {
            mbar_init(blk_full + 8 * s, 1 + (has_eta ? 32 : 0));
            mbar_init(blk_empty + 8 * s, C::NCW);
        }
        mbar_init(dead, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (warp > C::PW) return;

    //  A pattern: blocks (rows 0-7, c), (rows 8-15, c), (rows 0-7, c+8), (rows 8-15, c+8)
    //  B pattern: blocks (rows 0-7, c), (rows 0-7, c+8), (rows 8-15, c), (rows 8-15, c+8)
    const int rowA = (lane & 7) + 8 * ((lane >> 3) & 1), colA = 8 * (lane >> 4);
    const int rowB = (lane & 7) + 8 * (lane >> 4), colB = 8 * ((lane >> 3) & 1);
    const int g = lane >> 2, t4 = lane & 3;

    if (warp == C::PW) {
        // ------------------------------------------------------------ producer
        for (int L = 0; L < nblk; ++L) {
            const int s = L & (NB - 1);
            // (in the timeout test the warps release nothing: give up after the test's limit)
            if (L >= NB && !mbar_wait(blk_empty + 8 * s, ((L / NB) & 1) ^ 1, p.status, kSiteProducerEmpty,
                                      p.test_stall_ns ? p.test_stall_ns : kWaitLimitNs))
                break;
            const uint32_t full = blk_full + 8 * s, st = base + s * C::SLOT;
            if (has_eta) {
                const uint32_t ed = base + C::ETA_OFF + s * 256;
#pragma unroll
                for (int i = lane; i < 64; i += 32)
                    if (64 * L + i < T) cp_async_4(ed + 4 * i, p.eta + (size_t)bh * p.T + tb + 64 * L + i);
                cp_async_arrive_noinc(full);
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(full, (QSIDE ? 3 : 2) * C::BLK);
                if (QSIDE) tma_load_3d(st, tq, full, 0, tb + 64 * L, bh);
                tma_load_3d(st + C::BLK, tk, full, 0, tb + 64 * L, bh);
                tma_load_3d(st + 2 * C::BLK, tv, full, 0, tb + 64 * L, bh);
            }
            __syncwarp();
        }
        for (int L = nblk > NB ? nblk - NB : 0; L < nblk; ++L)
            if (!mbar_wait(blk_full + 8 * (L & (NB - 1)), (L / NB) & 1, p.status, kSiteDrain)) break;
        return;
    }

    // ------------------------------------------------------------ compute warp
    // MAP: warps 0 .. D/16-1 hold columns of A, the others columns of B
    const int part = MAP ? warp / (D / 16) : 0;
    const int w = MAP ? warp % (D / 16) : warp, col0 = 16 * w;
    const bool zero_v = MAP && part == 0;  // the columns of A see labels V = 0
    float wacc[NJ][4];  // W^T[col0+g (+8)][8j+2t4 .. +1]
    if constexpr (MAP) {
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                wacc[j][i] = (part == 0 && 8 * j + 2 * t4 + (i & 1) == col0 + g + 8 * (i >> 1)) ? 1.f : 0.f;
    } else {
        const float *W0 = seg == 0 ? p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * D * D
                                   : p.Wst + ((size_t)bh * (p.nsplit - 1) + seg - 1) * D * D;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int r = 8 * j + 2 * t4;
            wacc[j][0] = W0[(size_t)r * D + col0 + g];
            wacc[j][1] = W0[(size_t)(r + 1) * D + col0 + g];
            wacc[j][2] = W0[(size_t)r * D + col0 + g + 8];
            wacc[j][3] = W0[(size_t)(r + 1) * D + col0 + g + 8];
        }
    }
    // bf16 W (the chunk's start weights): for k-tile kk, words 4kk..4kk+3 are
    // (tile 2kk rows g, g+8), (tile 2kk+1 rows g, g+8)
    uint32_t wb[2 * NJ];
    auto convert = [&]() {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int o = 4 * (j >> 1) + 2 * (j & 1);
            wb[o] = pack_bf16(wacc[j][0], wacc[j][1]);
            wb[o + 1] = pack_bf16(wacc[j][2], wacc[j][3]);
        }
    };
    convert();

    uint32_t offA[NK], offB[NK];
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
        offA[kk] = boff<D>(rowA, 16 * kk + colA);
        offB[kk] = boff<D>(rowB, 16 * kk + colB);
    }
    const uint32_t offV = boff<D>(rowB, col0 + colB);
    [[maybe_unused]] const uint32_t offQz = boff<D>(rowA, col0 + colA);
    // inner norm scale / shift of this lane's columns: as rows of E^T (col0 + g,
    // col0 + g + 8) and as columns of Z (col0 + 8hh + 2t4 + j)
    [[maybe_unused]] float ge[2] = {}, be[2] = {}, gz[2][2] = {}, bz[2][2] = {};
    if constexpr (LN) {
        const float *gm = p.ln_gamma + (size_t)(bh % p.H) * D, *bt = p.ln_beta + (size_t)(bh % p.H) * D;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            ge[r] = gm[col0 + g + 8 * r];
            be[r] = bt[col0 + g + 8 * r];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                gz[r][j] = gm[col0 + 8 * r + 2 * t4 + j];
                bz[r][j] = bt[col0 + 8 * r + 2 * t4 + j];
            }
        }
    }
    float2 *const red = reinterpret_cast<float2 *>(gbase + C::RED_OFF);  // [3][NCW][16]

    // fragments of chunk (L, Q) from block slot L % NB (the block has landed)
    auto load = [&](auto qc, Frag<D> &F, int L) {
        constexpr int Q = decltype(qc)::value;
        const uint32_t st = base + (L & (NB - 1)) * C::SLOT + 16 * Q * C::RB;
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
            ldsm_x4(st + C::BLK + offB[kk], F.kB[kk][0], F.kB[kk][1], F.kB[kk][2], F.kB[kk][3]);
            ldsm_x4_t(st + C::BLK + offA[kk], F.kT[kk][0], F.kT[kk][1], F.kT[kk][2], F.kT[kk][3]);
            if (QSIDE) ldsm_x4(st + offA[kk], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3]);
        }
        if (zero_v)
            F.vv[0][0] = F.vv[0][1] = F.vv[1][0] = F.vv[1][1] = 0u;
        else
            ldsm_x4_t(st + 2 * C::BLK + offV, F.vv[0][0], F.vv[0][1], F.vv[1][0], F.vv[1][1]);
        if constexpr (LN) {
            ldsm_x4_t(st + C::BLK + offV, F.kc[0][0], F.kc[0][1], F.kc[1][0], F.kc[1][1]);
            ldsm_x4(st + offQz, F.qz[0], F.qz[1], F.qz[2], F.qz[3]);
        }
        if constexpr (DELTA)
#pragma unroll
            for (int kk = 0; kk < NK; ++kk)
                ldsm_x4(st + C::BLK + offA[kk], F.ka[kk][0], F.ka[kk][1], F.ka[kk][2], F.ka[kk][3]);
        if (has_eta) {
            const float *e = reinterpret_cast<const float *>(gbase + C::ETA_OFF + (L & (NB - 1)) * 256) +
                             16 * Q + 2 * t4;
            F.et[0][0] = e[0];
            F.et[0][1] = e[1];
            F.et[1][0] = e[8];
            F.et[1][1] = e[9];
        } else {
            F.et[0][0] = F.et[0][1] = F.et[1][0] = F.et[1][1] = p.eta_scalar;
        }
    };

    bool vis[2][4];  // causal visibility of (query g + 8(i>>1), key 8nt + 2t4 + (i&1))
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) vis[nt][i] = !p.causal || (8 * nt + 2 * t4 + (i & 1)) <= g + 8 * (i >> 1);
    __nv_bfloat16 *const zlane =
        QSIDE ? p.z + ((size_t)bh * p.T + tb) * D + (size_t)g * D + col0 + 2 * t4 : nullptr;

    bool next_ready = false;  // the next block has landed (tested in chunk 2 of a block)

    // Inner norm: sums over all d columns of per-token partials (a, b).  Layout of E^T
    // (this lane: tokens 8nt + 2t4 + j, two columns): reduce over the lanes of equal t4,
    // then over the warps through shared-memory buffer `buf`.
    [[maybe_unused]] auto tok_sums_e = [&](int buf, float (&a)[2][2], float (&b)[2][2]) {
        // reduce-scatter over the 8 lanes of equal t4: value k = 4 nt + 2 j + stat ends in
        // the lane whose bits (4, 3, 2) are the bits of k
        float v[8];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                v[4 * nt + 2 * j] = a[nt][j];
                v[4 * nt + 2 * j + 1] = b[nt][j];
            }
        const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
        float u[4], x[2];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            u[i] = (b4 ? v[4 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[4 + i], 16);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            x[i] = (b3 ? u[2 + i] : u[i]) + __shfl_xor_sync(0xffffffffu, b3 ? u[i] : u[2 + i], 8);
        const float tot = (b2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, b2 ? x[0] : x[1], 4);
        float *redf = reinterpret_cast<float *>(red);
        redf[((buf * C::NCW + w) * 16 + 8 * b4 + 2 * t4 + b3) * 2 + b2] = tot;
        bar_compute(C::NCW * 32);
        // tokens 8nt + 2t4 and 8nt + 2t4 + 1 sit side by side: one 16-byte load per warp
        // and token pair, summed over the warps two floats at a time
        const float4 *red4 = reinterpret_cast<const float4 *>(red);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float4 t = red4[(buf * C::NCW * 16 + 8 * nt + 2 * t4) >> 1];
            float2 s0 = make_float2(t.x, t.y), s1 = make_float2(t.z, t.w);
#pragma unroll
            for (int ww = 1; ww < C::NCW; ++ww) {
                t = red4[((buf * C::NCW + ww) * 16 + 8 * nt + 2 * t4) >> 1];
                s0 = __fadd2_rn(s0, make_float2(t.x, t.y));
                s1 = __fadd2_rn(s1, make_float2(t.z, t.w));
            }
            a[nt][0] = s0.x;
            b[nt][0] = s0.y;
            a[nt][1] = s1.x;
            b[nt][1] = s1.y;
        }
    };

    // one chunk (L, Q) on fragments F; fetches chunk (L, Q+1) or (L+1, 0) into Fn.
    // FULL: the chunk has 16 tokens (no bounds masks).  Returns false when there
    // is no next chunk (or a wait gave up).
    auto chunk = [&](auto qc, auto fullc, Frag<D> &F, Frag<D> &Fn, int L) -> bool {
        constexpr int Q = decltype(qc)::value;
        constexpr bool FULL = decltype(fullc)::value;
        const int t0 = 64 * L + 16 * Q;
        const int c = FULL ? 16 : T - t0;
        // E^T = W^T K^T - V^T.  ONE: a single accumulator per n-tile that starts at
        // -V^T (fewer instructions, a deeper product chain: the map role has a second
        // warp on each SM sub-partition to hide it); otherwise two interleaved
        // accumulators with V subtracted afterwards (shorter chain for the lone warp)
        constexpr bool ONE = true;
        float e[2][2][4] = {};
        [[maybe_unused]] float sc[2][4] = {}, zc[2][4] = {};
        if constexpr (ONE && !LN) {  // (the inner norm takes V after the norm)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t vw = F.vv[nt][i >> 1];
                    e[0][nt][i] = -((i & 1) ? bf16_hi(vw) : bf16_lo(vw));
                }
        }
#pragma unroll
        for (int kk = 0; kk < NK && !DOT; ++kk) {
            mma_bf16(e[ONE ? 0 : kk & 1][0], wb[4 * kk], wb[4 * kk + 1], wb[4 * kk + 2], wb[4 * kk + 3],
                     F.kB[kk][0], F.kB[kk][1]);
            mma_bf16(e[ONE ? 0 : kk & 1][1], wb[4 * kk], wb[4 * kk + 1], wb[4 * kk + 2], wb[4 * kk + 3],
                     F.kB[kk][2], F.kB[kk][3]);
        }
#pragma unroll
        for (int kk = 0; kk < NK && QSIDE; ++kk) {  // S = Q K^T (off the serial chain)
            mma_bf16(sc[0], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3], F.kB[kk][0], F.kB[kk][1]);
            mma_bf16(sc[1], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3], F.kB[kk][2], F.kB[kk][3]);
        }
        [[maybe_unused]] float gk[2][4] = {};  // delta rule: K K^T of the chunk (inputs only)
#pragma unroll
        for (int kk = 0; kk < NK && DELTA; ++kk) {
            mma_bf16(gk[0], F.ka[kk][0], F.ka[kk][1], F.ka[kk][2], F.ka[kk][3], F.kB[kk][0], F.kB[kk][1]);
            mma_bf16(gk[1], F.ka[kk][0], F.ka[kk][1], F.ka[kk][2], F.ka[kk][3], F.kB[kk][2], F.kB[kk][3]);
        }
        // next chunk's fragments: inside a block the load is unconditional (reads of
        // the ring past the sequence end stay in bounds and are never used), so the
        // chunk body stays one basic block; crossing into the next block waits for it
        const bool more = t0 + 16 < T;
        bool alive = true;  // false: a wait gave up
        if constexpr (Q < 3) {
            load(std::integral_constant<int, Q + 1>{}, Fn, L);
            // test for the next block a chunk ahead (non-blocking): the result is
            // read in the block's last chunk, so the test's latency is hidden
            if constexpr (Q == 2)
                next_ready = mbar_test_wait(blk_full + 8 * ((L + 1) & (NB - 1)), ((L + 1) / NB) & 1);
        } else {
            // the block's last chunk: release the block, wait for the next one if there is
            // one, and load its first fragments whether or not it exists (the ring slot is
            // always in bounds; unused past the end).  Without a branch around this part
            // the chunk body stays one basic block, which measured 7% faster than the
            // conditional form; a wait that gives up is reported through the return value
            __syncwarp();
            if (lane == 0) mbar_arrive(blk_empty + 8 * (L & (NB - 1)));
            alive = next_ready || !more ||
                    mbar_wait(blk_full + 8 * ((L + 1) & (NB - 1)), ((L + 1) / NB) & 1, p.status, kSiteConsumerFull);
            if constexpr (LN) alive = bar_compute_and(C::NCW * 32, alive);  // all warps go on, or none
            load(std::integral_constant<int, 0>{}, Fn, L + 1);
        }
        if constexpr (LN) {  // Z = Q W first: the tensor pipe works through the norm's exchanges
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                mma_bf16(zc[0], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3], wb[4 * kk], wb[4 * kk + 2]);
                mma_bf16(zc[1], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3], wb[4 * kk + 1],
                         wb[4 * kk + 3]);
            }
        }
        if constexpr (LN) {
            // e currently holds Y^T = (K W)^T.  Elements (nt, 2r + j), j = 0, 1, are tokens
            // 8nt + 2t4 + j of row col0 + g + 8r: pairs over j share the token statistics, so
            // the norm runs on paired fp32 instructions.  Forward statistics first.
            auto yp = [&](int nt, int r) { return make_float2(e[0][nt][2 * r], e[0][nt][2 * r + 1]); };
            const float2 invd = make_float2(1.f / D, 1.f / D), m1 = make_float2(-1.f, -1.f);
            float a[2][2], b[2][2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 y0 = yp(nt, 0), y1 = yp(nt, 1);
                const float2 s2 = __fadd2_rn(y0, y1), q2 = __ffma2_rn(y0, y0, __fmul2_rn(y1, y1));
                a[nt][0] = s2.x;
                a[nt][1] = s2.y;
                b[nt][0] = q2.x;
                b[nt][1] = q2.y;
            }
            tok_sums_e(0, a, b);
            float2 rs[2], mr[2];  // per nt: 1 / sigma and -mu / sigma of tokens j = 0, 1
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 mu = __fmul2_rn(make_float2(a[nt][0], a[nt][1]), invd);
                const float2 var = __ffma2_rn(__fmul2_rn(mu, m1), mu, __fmul2_rn(make_float2(b[nt][0], b[nt][1]), invd));
                rs[nt] = make_float2(rsqrtf(fmaxf(var.x, 0.f) + p.ln_eps), rsqrtf(fmaxf(var.y, 0.f) + p.ln_eps));
                mr[nt] = __fmul2_rn(__fmul2_rn(mu, m1), rs[nt]);
            }
            // residual through the norm, e = k + LN(y) - v, and g = gamma e
            float2 yh[2][2], gg[2][2];  // [nt][r]
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    yh[nt][r] = __ffma2_rn(yp(nt, r), rs[nt], mr[nt]);
                    const float2 kv = make_float2(bf16_lo(F.kc[nt][r]), bf16_hi(F.kc[nt][r]));
                    const float2 vv = make_float2(bf16_lo(F.vv[nt][r]), bf16_hi(F.vv[nt][r]));
                    const float2 kb = __ffma2_rn(vv, m1, __fadd2_rn(kv, make_float2(be[r], be[r])));
                    const float2 g2 = make_float2(ge[r], ge[r]);
                    gg[nt][r] = __fmul2_rn(g2, __ffma2_rn(g2, yh[nt][r], kb));
                }
            // backward statistics: means of g and g * yh over the row
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 s2 = __fadd2_rn(gg[nt][0], gg[nt][1]);
                const float2 q2 = __ffma2_rn(gg[nt][0], yh[nt][0], __fmul2_rn(gg[nt][1], yh[nt][1]));
                a[nt][0] = s2.x;
                a[nt][1] = s2.y;
                b[nt][0] = q2.x;
                b[nt][1] = q2.y;
            }
            tok_sums_e(1, a, b);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float2 na = __fmul2_rn(make_float2(a[nt][0], a[nt][1]), __fmul2_rn(invd, m1));
                const float2 bd = __fmul2_rn(make_float2(b[nt][0], b[nt][1]), invd);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    // (g - mean g - yh mean(g yh)) / sigma
                    const float2 x = __fmul2_rn(__ffma2_rn(__fmul2_rn(yh[nt][r], m1), bd, __fadd2_rn(gg[nt][r], na)), rs[nt]);
                    e[0][nt][2 * r] = x.x;
                    e[0][nt][2 * r + 1] = x.y;
                }
            }
        }
        if constexpr (DELTA) {
            // e holds R^T = (K W - V)^T at the chunk's start weights.  Coupling of the
            // chunk, A[t][s] = (k_t . k_s) eta_s for s < t, stored as [s][t] in this
            // warp's 1 KB: the accumulator element (t = g + 8(i>>1), s = 8nt + 2t4 + (i&1))
            float *As = reinterpret_cast<float *>(gbase + C::DA_OFF) + warp * 256;
            __syncwarp();  // the previous chunk's reads of As are done
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = g + 8 * (i >> 1), sk = 8 * nt + 2 * t4 + (i & 1);
                    As[sk * 16 + t] = (sk < t && (FULL || t < c)) ? gk[nt][i] * F.et[nt][i & 1] : 0.f;
                }
            __syncwarp();
            // forward substitution: once token s's residual is final (columns g, g + 8 in
            // lane t4 = (s mod 8) / 2 of each row group), every token t of the lane loses
            // A[t][s] e_s (zero unless t > s)
#pragma unroll
            for (int si = 0; si < 15; ++si) {
                const int src = (lane & ~3) | ((si & 7) >> 1);
                const float v0 = __shfl_sync(0xffffffffu, e[0][si >> 3][si & 1], src);
                const float v1 = __shfl_sync(0xffffffffu, e[0][si >> 3][2 + (si & 1)], src);
                const float2 a0 = *reinterpret_cast<const float2 *>(As + si * 16 + 2 * t4);
                const float2 a1 = *reinterpret_cast<const float2 *>(As + si * 16 + 8 + 2 * t4);
                e[0][0][0] = fmaf(-a0.x, v0, e[0][0][0]);
                e[0][0][1] = fmaf(-a0.y, v0, e[0][0][1]);
                e[0][0][2] = fmaf(-a0.x, v1, e[0][0][2]);
                e[0][0][3] = fmaf(-a0.y, v1, e[0][0][3]);
                e[0][1][0] = fmaf(-a1.x, v0, e[0][1][0]);
                e[0][1][1] = fmaf(-a1.y, v0, e[0][1][1]);
                e[0][1][2] = fmaf(-a1.x, v1, e[0][1][2]);
                e[0][1][3] = fmaf(-a1.y, v1, e[0][1][3]);
            }
        }
        // -Et^T as an A fragment
        float ne[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float r = e[0][nt][i];
                if constexpr (!ONE) {
                    const uint32_t vw = F.vv[nt][i >> 1];
                    r += e[1][nt][i] - ((i & 1) ? bf16_hi(vw) : bf16_lo(vw));
                }
                ne[nt][i] = (FULL || (8 * nt + 2 * t4 + (i & 1)) < c) ? -F.et[nt][i & 1] * r : 0.f;
            }
        const uint32_t ea0 = pack_bf16(ne[0][0], ne[0][1]), ea1 = pack_bf16(ne[0][2], ne[0][3]);
        const uint32_t ea2 = pack_bf16(ne[1][0], ne[1][1]), ea3 = pack_bf16(ne[1][2], ne[1][3]);
#pragma unroll
        for (int j2 = 0; j2 < NK; ++j2) {  // W^T += (-Et^T) K
            mma_bf16(wacc[2 * j2], ea0, ea1, ea2, ea3, F.kT[j2][0], F.kT[j2][1]);
            mma_bf16(wacc[2 * j2 + 1], ea0, ea1, ea2, ea3, F.kT[j2][2], F.kT[j2][3]);
        }
        if constexpr (QSIDE) {
            // Z = Q W + (mask .* S)(-Et), masked scores as an A fragment from registers
    #pragma unroll
            for (int kk = 0; kk < NK && !LN; ++kk) {
                mma_bf16(zc[0], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3], wb[4 * kk], wb[4 * kk + 2]);
                mma_bf16(zc[1], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3], wb[4 * kk + 1],
                         wb[4 * kk + 3]);
            }
            float sm[2][4];
    #pragma unroll
            for (int nt = 0; nt < 2; ++nt)
    #pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool keep = vis[nt][i] && (FULL || (8 * nt + 2 * t4 + (i & 1)) < c);
                    sm[nt][i] = keep ? sc[nt][i] : 0.f;
                }
            mma_bf16(zc[0], pack_bf16(sm[0][0], sm[0][1]), pack_bf16(sm[0][2], sm[0][3]),
                     pack_bf16(sm[1][0], sm[1][1]), pack_bf16(sm[1][2], sm[1][3]), ea0, ea2);
            mma_bf16(zc[1], pack_bf16(sm[0][0], sm[0][1]), pack_bf16(sm[0][2], sm[0][3]),
                     pack_bf16(sm[1][0], sm[1][1]), pack_bf16(sm[1][2], sm[1][3]), ea1, ea3);
        }
        if constexpr (LN) {
            // zc holds Q W_t: z = q + LN(q W_t) per token (rows g, g + 8 of Z; elements
            // (hh, 2r + j) are columns col0 + 8hh + 2t4 + j of row g + 8r)
            float v[4];  // (sum, sum of squares) of rows g, g + 8 over this lane's 4 columns
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float2 z0 = make_float2(zc[0][2 * r], zc[0][2 * r + 1]);
                const float2 z1 = make_float2(zc[1][2 * r], zc[1][2 * r + 1]);
                const float2 s2 = __fadd2_rn(z0, z1), q2 = __ffma2_rn(z0, z0, __fmul2_rn(z1, z1));
                v[2 * r] = s2.x + s2.y;
                v[2 * r + 1] = q2.x + q2.y;
            }
            // reduce-scatter over the row's 4 lanes: value 2r + stat ends in lane t4 = 2r + stat
            const bool c1 = (t4 >> 1) & 1, c0 = t4 & 1;
            float u[2];
#pragma unroll
            for (int k = 0; k < 2; ++k)
                u[k] = (c1 ? v[2 + k] : v[k]) + __shfl_xor_sync(0xffffffffu, c1 ? v[k] : v[2 + k], 2);
            const float tot = (c0 ? u[1] : u[0]) + __shfl_xor_sync(0xffffffffu, c0 ? u[0] : u[1], 1);
            reinterpret_cast<float *>(red)[((2 * C::NCW + w) * 16 + g + 8 * c1) * 2 + c0] = tot;
            bar_compute(C::NCW * 32);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float2 sm = red[(2 * C::NCW) * 16 + g + 8 * r];
#pragma unroll
                for (int ww = 1; ww < C::NCW; ++ww) sm = __fadd2_rn(sm, red[(2 * C::NCW + ww) * 16 + g + 8 * r]);
                const float mu = sm.x * (1.f / D);
                const float rs = rsqrtf(fmaxf(sm.y * (1.f / D) - mu * mu, 0.f) + p.ln_eps);
                const float2 rs2 = make_float2(rs, rs), mr2 = make_float2(-mu * rs, -mu * rs);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float2 zh = __ffma2_rn(make_float2(zc[hh][2 * r], zc[hh][2 * r + 1]), rs2, mr2);
                    const float2 qv = make_float2(bf16_lo(F.qz[2 * hh + r]), bf16_hi(F.qz[2 * hh + r]));
                    const float2 zo = __fadd2_rn(qv, __ffma2_rn(make_float2(gz[hh][0], gz[hh][1]), zh,
                                                              make_float2(bz[hh][0], bz[hh][1])));
                    zc[hh][2 * r] = zo.x;
                    zc[hh][2 * r + 1] = zo.y;
                }
            }
        }
        convert();
        if constexpr (QSIDE) {
            __nv_bfloat16 *zb = zlane + (size_t)t0 * D;
    #pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (FULL || g < c)
                    *reinterpret_cast<uint32_t *>(zb + 8 * hh) = pack_bf16(zc[hh][0], zc[hh][1]);
                if (FULL || g + 8 < c)
                    *reinterpret_cast<uint32_t *>(zb + 8 * D + 8 * hh) = pack_bf16(zc[hh][2], zc[hh][3]);
            }
        }
        return more && alive;
    };
    // the four chunks of block L; FULL: the block holds 64 tokens (no bounds masks)
    auto block = [&](auto fullc, Frag<D> &FA, Frag<D> &FB, int L) -> bool {
        using I0 = std::integral_constant<int, 0>;
        using I1 = std::integral_constant<int, 1>;
        using I2 = std::integral_constant<int, 2>;
        using I3 = std::integral_constant<int, 3>;
        if constexpr (decltype(fullc)::value) {
            // a full block's first three chunks always have a successor inside the block and
            // never wait: the four run in sequence, with no branch between them
            chunk(I0{}, fullc, FA, FB, L);
            chunk(I1{}, fullc, FB, FA, L);
            chunk(I2{}, fullc, FA, FB, L);
            return chunk(I3{}, fullc, FB, FA, L);
        } else {
            return chunk(I0{}, fullc, FA, FB, L) && chunk(I1{}, fullc, FB, FA, L) && chunk(I2{}, fullc, FA, FB, L) &&
                   chunk(I3{}, fullc, FB, FA, L);
        }
    };

    bool first = nblk > 0 && (p.test_stall_ns ? mbar_wait(dead, 0, p.status, kSiteConsumerFull, p.test_stall_ns)
                                                : mbar_wait(blk_full, 0, p.status, kSiteConsumerFull));
    if constexpr (LN)  // the chunks meet at named barriers: every compute warp starts, or none
        if (nblk > 0) first = bar_compute_and(C::NCW * 32, first);
    if (first) {
        Frag<D> FA, FB;
        load(std::integral_constant<int, 0>{}, FA, 0);
        for (int L = 0;; ++L) {  // two fragment sets alternate: no register copies
            const bool ok = 64 * L + 64 <= T ? block(std::true_type{}, FA, FB, L) : block(std::false_type{}, FA, FB, L);
            if (!ok) break;
        }
    }

    float *Wo = nullptr;
    if (ROLE == kRoleMap)  // map of segment seg (1 .. nsplit-2)
        Wo = p.maps + (((size_t)bh * (p.nsplit - 2) + seg - 1) * 2 + part) * D * D;
    else if (ROLE == kRoleChain)  // end of segment seg = start of segment seg + 1
        Wo = p.Wst + ((size_t)bh * (p.nsplit - 1) + seg) * D * D;
    else if (p.W_out && seg == p.nsplit - 1)
        Wo = p.W_out + (size_t)bh * D * D;
    if (Wo) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int r = 8 * j + 2 * t4;
            Wo[(size_t)r * D + col0 + g] = wacc[j][0];
            Wo[(size_t)(r + 1) * D + col0 + g] = wacc[j][1];
            Wo[(size_t)r * D + col0 + g + 8] = wacc[j][2];
            Wo[(size_t)(r + 1) * D + col0 + g + 8] = wacc[j][3];
        }
    }
}

// Output units: CTA u serves chain u / nseg, segment seg0 + u % nseg.
template <int D, int VAR>
__global__ void __launch_bounds__(B16Cfg<D, false>::THREADS, 1)
    ttt_linear_b16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv, const B16Params p)
{
    b16_unit<D, kRoleOut, VAR>(&tq, &tk, &tv, p, blockIdx.x / p.nseg, p.seg0 + blockIdx.x % p.nseg);
}

// The work before a split run's later segments: CTAs 0 .. BH-1 run the state chain
// of each chain's first segment, the others the affine maps of segments
// 1 .. nsplit-2 (chain (u - BH) / (nsplit - 2)).
template <int D, int VAR>
__global__ void __launch_bounds__(B16Cfg<D, true>::THREADS, 1)
    ttt_linear_b16_prep_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                               const __grid_constant__ CUtensorMap tv, const B16Params p)
{
    const int u = blockIdx.x;
    if (u < p.BH)
        b16_unit<D, kRoleChain, VAR>(&tq, &tk, &tv, p, u, 0);
    else
        b16_unit<D, kRoleMap, VAR>(&tq, &tk, &tv, p, (u - p.BH) / (p.nsplit - 2), 1 + (u - p.BH) % (p.nsplit - 2));
}

template <int D, bool PREP>
int launch_b16_t(const LinearArgs &a, const B16Params &p, int units, const CUtensorMap *maps)
{
    using C = B16Cfg<D, PREP>;
    auto kern = PREP       ? (a.b == 1 ? ttt_linear_b16_prep_kernel<D, 3> : ttt_linear_b16_prep_kernel<D, 0>)
                : a.ln_gamma   ? ttt_linear_b16_kernel<D, 2>
                : a.loss       ? ttt_linear_b16_kernel<D, 1>
                : a.b == 1     ? ttt_linear_b16_kernel<D, 3>
                               : ttt_linear_b16_kernel<D, 0>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return -4;
    kern<<<units, C::THREADS, C::SMEM, a.stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

B16Params b16_params(const LinearArgs &a)
{
    B16Params p;
    p.BH = a.B * a.H;
    p.H = a.H;
    p.T = a.T;
    p.causal = a.b == 1 ? 1 : a.causal;  // one-token mini-batches: every query reads its own write
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W0 = a.W0;
    p.w0_bstride = a.w0_bstride;
    p.z = static_cast<__nv_bfloat16 *>(a.z);
    p.W_out = a.W_out;
    p.status = a.status;
    p.len0 = p.seg_len = ((a.T + 63) / 64) * 64;  // one unit per chain: the whole sequence
    p.nseg = 1;
    p.seg0 = 0;
    p.nsplit = 1;
    p.Wst = nullptr;
    p.maps = nullptr;
    p.ln_gamma = a.ln_gamma;
    p.ln_beta = a.ln_beta;
    p.ln_eps = a.ln_eps;
    p.test_stall_ns = a.test_stall_ns;
    return p;
}

template <bool PREP>
int launch_b16_d(const LinearArgs &a, const B16Params &p, int units, const CUtensorMap *maps)
{
    switch (a.d) {
    case 16: return launch_b16_t<16, PREP>(a, p, units, maps);
    case 32: return launch_b16_t<32, PREP>(a, p, units, maps);
    case 64: return launch_b16_t<64, PREP>(a, p, units, maps);
    default: return -2;
    }
}

}  // namespace

int launch_linear_b16(const LinearArgs &a)
{
    if (a.d > 64) return launch_linear_bf16(a);
    CUtensorMap maps[3];
    if (!encode_qkv(maps, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 64)) return -4;
    return launch_b16_d<false>(a, b16_params(a), a.B * a.H, maps);
}

int launch_linear_b16_segments(const LinearArgs &a, int nsplit, int len0, int seg_len, int seg0, int nseg,
                               bool prep, float *Wst, float *mapbuf, const CUtensorMap *maps)
{
    B16Params p = b16_params(a);
    p.len0 = len0;
    p.seg_len = seg_len;
    p.nseg = nseg;
    p.seg0 = seg0;
    p.nsplit = nsplit;
    p.Wst = Wst;
    p.maps = mapbuf;
    if (prep) return launch_b16_d<true>(a, p, a.B * a.H * (nsplit - 1), maps);
    return launch_b16_d<false>(a, p, a.B * a.H * nseg, maps);
}

}  // namespace ttt
