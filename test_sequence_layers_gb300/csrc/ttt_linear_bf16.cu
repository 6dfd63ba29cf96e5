// ttt_linear_bf16.cu -- TTT-Linear forward on sm_103a: bf16 operands, fp32
// accumulation, fp32 weight state.
//
// Per (batch, head) chain and per mini-batch with start weights W (row
// convention, f(x;W) = x W), the matrix form of the mini-batch step is
//     E  = K W - V                       residuals at the block's start weights
//     Et = diag(eta) E
//     Z  = Q W_cur - (mask .* (Q K^T)) Et  mask = lower triangle incl. diagonal
//                                          (causal) or all ones (non-causal)
//     W  <- W - K^T Et
// ("Learning to (Learn at Test Time)" walkthrough, section 1.2.2, dual form: a
// lower-triangular mask of zeros replaces the per-token gradients; gradients of
// all tokens at the previous block's W, outputs through the cumulative sum).
//
// Work split.  Column j of W, E and Z depends only on column j of W0 and V (plus
// the shared Q, K, eta), so each "chain warp" owns 16 output columns of the
// state and carries them through the whole sequence in registers, with no
// exchange between warps on the serial dependency.  The state is held as W^T
// (16 x d) in mma.sync accumulator fragments: the accumulator layout of W^T is
// at the same time the A operand of E^T = W^T K^T and the B operand of
// Z = Q W, and E^T's accumulator is the A operand of the update
// W^T += (-Et^T) K, so the serial chain E -> Et -> update never leaves
// registers.  A "score" warp computes mask .* (Q K^T) once per tile for all
// chain warps, and a producer warp streams the Q/K/V tiles with TMA (128-byte
// swizzle, conflict-free ldmatrix) through an NS-stage mbarrier pipeline; the
// per-token eta comes in with 4-byte cp.async on the same barriers.
//
// Why warp-level mma.sync and not tcgen05 here: the shapes on the serial chain
// are 16x16x64 and 16x64x16 per step, and every step depends on the previous
// one; a tcgen05 round trip (issue, commit, mbarrier, TMEM load, convert, shared
// store) per dependent product costs more than the whole step takes here.
#include <cuda.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"
#include "ttt_jobs.cuh"

namespace ttt {

template <int D>
struct LinCfg {
    static constexpr int NCW = D / 16;                 // chain warps, 16 columns each
    static constexpr int WARPS = NCW + 2;              // + score warp + producer warp
    static constexpr int THREADS = WARPS * 32;
    static constexpr int NS = 8;                       // pipeline stages
    static constexpr int RB = (D < 64 ? D : 64) * 2;   // bytes per row of a TMA box
    static constexpr int SUB = 16 * RB;                // bytes per box (16 rows)
    static constexpr int TILE = 16 * D * 2;            // bytes of a 16 x D tile
    static constexpr int TILE_A = ((TILE + 1023) / 1024) * 1024;
    static constexpr int SROW = 48;                    // padded row of a 16 x 16 bf16 tile
    static constexpr int S_OFF = 3 * TILE_A;           // scores (bf16 16 x 16)
    static constexpr int ETA_OFF = S_OFF + 16 * SROW;  // eta (16 fp32)
    static constexpr int STAGE = ((ETA_OFF + 64 + 1023) / 1024) * 1024;
    static constexpr int ZST_OFF = NS * STAGE;         // per-chain-warp output staging
    static constexpr int BAR_OFF = ZST_OFF + NCW * 16 * SROW;
    static constexpr int SMEM = BAR_OFF + 3 * NS * 8 + 1024;  // + base alignment slack
    static constexpr uint32_t SWM = RB == 128 ? 7u : (RB == 64 ? 3u : 1u);
};

// Byte offset of element (r, c) in a 16 x D bf16 tile written by TMA with the
// 32/64/128-byte swizzle matching the box row length (16-byte chunk index XOR
// the 128-byte line index).
template <int D>
__device__ __forceinline__ uint32_t toff(int r, int c)
{
    using C = LinCfg<D>;
    const int h = c >> 6, cc = c & 63;
    uint32_t a = static_cast<uint32_t>(r * C::RB + cc * 2);
    a ^= ((a >> 7) & C::SWM) << 4;
    return static_cast<uint32_t>(h * C::SUB) + a;
}

struct LinParams {
    int H, T, b, causal, dot;  // dot: negative dot-product loss (residual -V)
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    __nv_bfloat16 *z;
    float *W_out;
    int *status;
};

template <int D>
__global__ void __launch_bounds__(LinCfg<D>::THREADS, 1)
    ttt_linear_bf16_kernel(const __grid_constant__ CUtensorMap tq,
                           const __grid_constant__ CUtensorMap tk,
                           const __grid_constant__ CUtensorMap tv, const LinParams p)
{
    using C = LinCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const uint32_t bar_full = base + C::BAR_OFF;
    const uint32_t bar_ready = bar_full + 8 * C::NS;
    const uint32_t bar_empty = bar_ready + 8 * C::NS;
    const bool has_eta = p.eta != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar_full + 8 * s, 1 + (has_eta ? 32 : 0));
            mbar_init(bar_ready + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, C::NCW + 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // fragment address patterns (see the fragment maps in the file header)
    const int rowA = (lane & 7) + 8 * ((lane >> 3) & 1), colA = 8 * (lane >> 4);
    const int rowB = (lane & 7) + 8 * (lane >> 4), colB = 8 * ((lane >> 3) & 1);
    const int g = lane >> 2, t4 = lane & 3;

    if (warp == C::NCW + 1) {
        // ------------------------------------------------------------ producer
        JobIter it(p.T, p.b, p.causal);
        int jb = 0;
        for (; it.valid(); it.next(), ++jb) {
            const int s = jb % C::NS;
            const uint32_t ph = (jb / C::NS) & 1;
            if (jb >= C::NS && !mbar_wait(bar_empty + 8 * s, ph ^ 1, p.status, kSiteProducerEmpty))
                break;
            const Job J = it.get();
            const uint32_t st = base + s * C::STAGE;
            const uint32_t full = bar_full + 8 * s;
            if (has_eta) {
                if (J.kind != kOut && lane < J.c)
                    cp_async_4(st + C::ETA_OFF + 4 * lane, p.eta + (size_t)bh * p.T + J.t0 + lane);
                cp_async_arrive_noinc(full);
            }
            if (lane == 0) {
                const bool lq = J.kind != kUpd, lkv = J.kind != kOut;
                mbar_arrive_expect_tx(full, (uint32_t)((lq ? 1 : 0) + (lkv ? 2 : 0)) * C::TILE);
#pragma unroll
                for (int h = 0; h < (D + 63) / 64; ++h) {
                    if (lq) tma_load_3d(st + h * C::SUB, &tq, full, 64 * h, J.t0, bh);
                    if (lkv) {
                        tma_load_3d(st + C::TILE_A + h * C::SUB, &tk, full, 64 * h, J.t0, bh);
                        tma_load_3d(st + 2 * C::TILE_A + h * C::SUB, &tv, full, 64 * h, J.t0, bh);
                    }
                }
            }
            __syncwarp();
        }
        // make sure no copy is still landing in shared memory when the CTA ends
        for (int j = (jb > C::NS ? jb - C::NS : 0); j < jb; ++j)
            if (!mbar_wait(bar_full + 8 * (j % C::NS), (j / C::NS) & 1, p.status, kSiteDrain)) break;
        return;
    }

    if (warp == C::NCW) {
        // ---------------------------------------------------------- score warp
        JobIter it(p.T, p.b, p.causal);
        for (int jb = 0; it.valid(); it.next(), ++jb) {
            const int s = jb % C::NS;
            const uint32_t ph = (jb / C::NS) & 1;
            const Job J = it.get();
            if (!mbar_wait(bar_full + 8 * s, ph, p.status, kSiteConsumerFull)) break;
            const uint32_t st = base + s * C::STAGE;
            if (J.kind == kBoth) {
                float sc[2][4] = {};
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t a0, a1, a2, a3, b00, b01, b10, b11;
                    ldsm_x4(st + toff<D>(rowA, 16 * kk + colA), a0, a1, a2, a3);
                    ldsm_x4(st + C::TILE_A + toff<D>(rowB, 16 * kk + colB), b00, b01, b10, b11);
                    mma_bf16(sc[0], a0, a1, a2, a3, b00, b01);
                    mma_bf16(sc[1], a0, a1, a2, a3, b10, b11);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int tq_ = g + 8 * (i >> 1), ss = 8 * nt + 2 * t4 + (i & 1);
                        const bool keep = ss < J.c && (!p.causal || ss <= tq_);
                        if (!keep) sc[nt][i] = 0.f;
                    }
                stsm_x4(st + C::S_OFF + rowA * C::SROW + colA * 2, pack_bf16(sc[0][0], sc[0][1]),
                        pack_bf16(sc[0][2], sc[0][3]), pack_bf16(sc[1][0], sc[1][1]),
                        pack_bf16(sc[1][2], sc[1][3]));
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar_ready + 8 * s);
                mbar_arrive(bar_empty + 8 * s);
            }
        }
        return;
    }

    // -------------------------------------------------------------- chain warp
    constexpr int NJ = D / 8;  // 8-column tiles along d_in
    const int w = warp;
    const int col0 = 16 * w;   // first output column owned by this warp

    // W^T fragment: w_[j][0..1] = W^T[col0+g][8j+2t4 .. +1], w_[j][2..3] = row col0+g+8
    float wacc[NJ][4];
    {
        const float *W0 = p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * D * D;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int r = 8 * j + 2 * t4;
            wacc[j][0] = W0[(size_t)r * D + col0 + g];
            wacc[j][1] = W0[(size_t)(r + 1) * D + col0 + g];
            wacc[j][2] = W0[(size_t)r * D + col0 + g + 8];
            wacc[j][3] = W0[(size_t)(r + 1) * D + col0 + g + 8];
        }
    }
    uint32_t wst[NJ][2], wcur[NJ][2];  // bf16 W_start (for E) and W_current (for Z)
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        wst[j][0] = wcur[j][0] = pack_bf16(wacc[j][0], wacc[j][1]);
        wst[j][1] = wcur[j][1] = pack_bf16(wacc[j][2], wacc[j][3]);
    }
    const uint32_t zst = base + C::ZST_OFF + w * 16 * C::SROW;

    JobIter it(p.T, p.b, p.causal);
    for (int jb = 0; it.valid(); it.next(), ++jb) {
        const int s = jb % C::NS;
        const uint32_t ph = (jb / C::NS) & 1;
        const Job J = it.get();
        const uint32_t st = base + s * C::STAGE;
        const uint32_t tQ = st, tK = st + C::TILE_A, tV = st + 2 * C::TILE_A;
        if (!mbar_wait(bar_full + 8 * s, ph, p.status, kSiteConsumerFull)) break;

        const bool upd = J.kind != kOut, out = J.kind != kUpd;
        uint32_t ea0 = 0, ea1 = 0, ea2 = 0, ea3 = 0;  // -Et^T as an A fragment (16 cols x 16 tok)
        if (upd) {
            // E^T = W_start^T K^T - V^T (two accumulator chains shorten the dependency)
            float e[2][4] = {}, e2[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                if (p.dot) break;
                uint32_t b00, b01, b10, b11;
                ldsm_x4(tK + toff<D>(rowB, 16 * kk + colB), b00, b01, b10, b11);
                float(&acc)[2][4] = (kk & 1) ? e2 : e;
                mma_bf16(acc[0], wst[2 * kk][0], wst[2 * kk][1], wst[2 * kk + 1][0],
                         wst[2 * kk + 1][1], b00, b01);
                mma_bf16(acc[1], wst[2 * kk][0], wst[2 * kk][1], wst[2 * kk + 1][0],
                         wst[2 * kk + 1][1], b10, b11);
            }
            uint32_t vv[2][2];
            ldsm_x4_t(tV + toff<D>(rowB, col0 + colB), vv[0][0], vv[0][1], vv[1][0], vv[1][1]);
            const float *eta_s = reinterpret_cast<const float *>(gbase + s * C::STAGE + C::ETA_OFF);
            float ne[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int tok = 8 * nt + 2 * t4 + i;
                    const bool ok = tok < J.c;
                    const float et = has_eta ? eta_s[tok] : p.eta_scalar;
                    const float r0 = e[nt][i] + e2[nt][i] - (i ? bf16_hi(vv[nt][0]) : bf16_lo(vv[nt][0]));
                    const float r1 = e[nt][2 + i] + e2[nt][2 + i] -
                                     (i ? bf16_hi(vv[nt][1]) : bf16_lo(vv[nt][1]));
                    ne[nt][i] = ok ? -et * r0 : 0.f;
                    ne[nt][2 + i] = ok ? -et * r1 : 0.f;
                }
            ea0 = pack_bf16(ne[0][0], ne[0][1]);
            ea1 = pack_bf16(ne[0][2], ne[0][3]);
            ea2 = pack_bf16(ne[1][0], ne[1][1]);
            ea3 = pack_bf16(ne[1][2], ne[1][3]);
            // W^T += (-Et^T) K
#pragma unroll
            for (int j2 = 0; j2 < D / 16; ++j2) {
                uint32_t k0, k1, k2, k3;
                ldsm_x4_t(tK + toff<D>(rowA, 16 * j2 + colA), k0, k1, k2, k3);
                mma_bf16(wacc[2 * j2], ea0, ea1, ea2, ea3, k0, k1);
                mma_bf16(wacc[2 * j2 + 1], ea0, ea1, ea2, ea3, k2, k3);
            }
        }
        if (!mbar_wait(bar_ready + 8 * s, ph, p.status, kSiteConsumerReady)) break;
        if (out) {
            // Z = Q W_cur + (mask .* Q K^T) (-Et)
            float zc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(tQ + toff<D>(rowA, 16 * kk + colA), a0, a1, a2, a3);
                mma_bf16(zc[0], a0, a1, a2, a3, wcur[2 * kk][0], wcur[2 * kk + 1][0]);
                mma_bf16(zc[1], a0, a1, a2, a3, wcur[2 * kk][1], wcur[2 * kk + 1][1]);
            }
            if (J.kind == kBoth) {
                uint32_t s0, s1, s2, s3;
                ldsm_x4(st + C::S_OFF + rowA * C::SROW + colA * 2, s0, s1, s2, s3);
                mma_bf16(zc[0], s0, s1, s2, s3, ea0, ea2);
                mma_bf16(zc[1], s0, s1, s2, s3, ea1, ea3);
            }
            stsm_x4(zst + rowA * C::SROW + colA * 2, pack_bf16(zc[0][0], zc[0][1]),
                    pack_bf16(zc[0][2], zc[0][3]), pack_bf16(zc[1][0], zc[1][1]),
                    pack_bf16(zc[1][2], zc[1][3]));
            __syncwarp();
            const int r = lane >> 1, hf = lane & 1;
            if (r < J.c) {
                const uint4 val = lds128(zst + r * C::SROW + hf * 16);
                *reinterpret_cast<uint4 *>(p.z + ((size_t)bh * p.T + J.t0 + r) * D + col0 + 8 * hf) = val;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        if (upd) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                wcur[j][0] = pack_bf16(wacc[j][0], wacc[j][1]);
                wcur[j][1] = pack_bf16(wacc[j][2], wacc[j][3]);
            }
        }
        if (J.last_of_mb) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                wst[j][0] = wcur[j][0];
                wst[j][1] = wcur[j][1];
            }
        }
    }

    if (p.W_out) {
        float *Wo = p.W_out + (size_t)bh * D * D;
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

template <int D>
static int launch_t(const LinearArgs &a, const CUtensorMap *maps)
{
    using C = LinCfg<D>;
    auto kern = ttt_linear_bf16_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
        return -4;
    LinParams p;
    p.H = a.H;
    p.T = a.T;
    p.b = a.b;
    p.causal = a.causal;
    p.dot = a.loss;
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W0 = a.W0;
    p.w0_bstride = a.w0_bstride;
    p.z = static_cast<__nv_bfloat16 *>(a.z);
    p.W_out = a.W_out;
    p.status = a.status;
    kern<<<a.B * a.H, C::THREADS, C::SMEM, a.stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_linear_bf16(const LinearArgs &a)
{
    CUtensorMap maps[3];
    if (!encode_qkv(maps, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 16)) return -4;
    switch (a.d) {
    case 16: return launch_t<16>(a, maps);
    case 32: return launch_t<32>(a, maps);
    case 64: return launch_t<64>(a, maps);
    case 128: return launch_t<128>(a, maps);
    default: return -2;
    }
}

}  // namespace ttt
