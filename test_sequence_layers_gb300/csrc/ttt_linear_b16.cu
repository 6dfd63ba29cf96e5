// ttt_linear_b16.cu -- TTT-Linear forward specialised to mini-batches of 16
// tokens (the mini-batch size the walkthrough reports for all its experiments,
// "Learning to (Learn at Test Time)", section 1.2.2 / 4.1), bf16 operands, fp32
// accumulation and fp32 weight state, d in {16, 32, 64}.
//
// The algebra is that of ttt_linear_bf16.cu (dual form of one mini-batch:
// E = K W - V, Z = Q W - (mask .* Q K^T) diag(eta) E, W -= K^T diag(eta) E, with W^T
// held as mma.sync accumulators, 16 output columns per warp).  With b = 16 every
// 16-token chunk is exactly one mini-batch, which allows a leaner schedule:
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
#include <cuda.h>

#include <type_traits>

#include "ttt_device.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

template <int D>
struct B16Cfg {
    static constexpr int NCW = D / 16;               // compute warps, 16 output columns each
    static constexpr int PW = NCW;                   // producer warp
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int NJ = D / 8, NK = D / 16;
    static constexpr int NB = 4;                     // 64-token blocks in flight
    static constexpr int RB = 2 * D;                 // bytes per token row
    static constexpr int BLK = 64 * RB;              // one tensor's 64-token block
    static constexpr int SLOT = ((3 * BLK + 1023) / 1024) * 1024;  // Q, K, V of one block
    static constexpr int ETA_OFF = NB * SLOT;        // 64 fp32 per block
    static constexpr int BAR_OFF = ETA_OFF + NB * 256;
    static constexpr int SMEM = BAR_OFF + 2 * NB * 8 + 1024;
    static constexpr uint32_t SWM = RB == 128 ? 7u : (RB == 64 ? 3u : 1u);
};

// Offset of element (r, c) inside a 64-token block written by TMA with the swizzle
// of its row length.  For r = 16q + r0 the swizzle key does not depend on q, so
// offsets of a chunk are this per-lane value plus 16 q RB.
template <int D>
__device__ __forceinline__ uint32_t boff(int r, int c)
{
    uint32_t a = static_cast<uint32_t>(r * B16Cfg<D>::RB + c * 2);
    return a ^ (((a >> 7) & B16Cfg<D>::SWM) << 4);
}

template <int D>
struct Frag {
    uint32_t kB[D / 16][4];  // K as the B operand of E^T = W^T K^T and of S
    uint32_t kT[D / 16][4];  // K as the B operand of the update (transposed load)
    uint32_t qa[D / 16][4];  // Q as the A operand of Z = Q W
    uint32_t vv[2][2];       // V^T in accumulator layout
    float et[2][2];          // eta of tokens 8nt + 2t4 + i of the chunk
};

struct B16Params {
    int H, T, causal;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    __nv_bfloat16 *z;
    float *W_out;
    int *status;
};

template <int D>
__global__ void __launch_bounds__(B16Cfg<D>::THREADS, 1)
    ttt_linear_b16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv, const B16Params p)
{
    using C = B16Cfg<D>;
    constexpr int NJ = C::NJ, NK = C::NK, NB = C::NB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x, T = p.T;
    const int nblk = (T + 63) >> 6;
    const bool has_eta = p.eta != nullptr;

    const uint32_t blk_full = base + C::BAR_OFF;      // block landed (producer -> warps)
    const uint32_t blk_empty = blk_full + 8 * NB;     // block released (warps -> producer)
    if (threadIdx.x == 0) {
        for (int s = 0; s < NB; ++s) {
            mbar_init(blk_full + 8 * s, 1 + (has_eta ? 32 : 0));
            mbar_init(blk_empty + 8 * s, C::NCW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    //  A pattern: blocks (rows 0-7, c), (rows 8-15, c), (rows 0-7, c+8), (rows 8-15, c+8)
    //  B pattern: blocks (rows 0-7, c), (rows 0-7, c+8), (rows 8-15, c), (rows 8-15, c+8)
    const int rowA = (lane & 7) + 8 * ((lane >> 3) & 1), colA = 8 * (lane >> 4);
    const int rowB = (lane & 7) + 8 * (lane >> 4), colB = 8 * ((lane >> 3) & 1);
    const int g = lane >> 2, t4 = lane & 3;

    if (warp == C::PW) {
        // ------------------------------------------------------------ producer
        for (int L = 0; L < nblk; ++L) {
            const int s = L & (NB - 1);
            if (L >= NB && !mbar_wait(blk_empty + 8 * s, ((L / NB) & 1) ^ 1, p.status, kSiteProducerEmpty))
                break;
            const uint32_t full = blk_full + 8 * s, st = base + s * C::SLOT;
            if (has_eta) {
                const uint32_t ed = base + C::ETA_OFF + s * 256;
#pragma unroll
                for (int i = lane; i < 64; i += 32)
                    if (64 * L + i < T) cp_async_4(ed + 4 * i, p.eta + (size_t)bh * T + 64 * L + i);
                cp_async_arrive_noinc(full);
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(full, 3 * C::BLK);
                tma_load_3d(st, &tq, full, 0, 64 * L, bh);
                tma_load_3d(st + C::BLK, &tk, full, 0, 64 * L, bh);
                tma_load_3d(st + 2 * C::BLK, &tv, full, 0, 64 * L, bh);
            }
            __syncwarp();
        }
        for (int L = nblk > NB ? nblk - NB : 0; L < nblk; ++L)
            if (!mbar_wait(blk_full + 8 * (L & (NB - 1)), (L / NB) & 1, p.status, kSiteDrain)) break;
        return;
    }

    // ------------------------------------------------------------ compute warp
    const int w = warp, col0 = 16 * w;
    float wacc[NJ][4];  // W^T[col0+g (+8)][8j+2t4 .. +1]
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

    // fragments of chunk (L, Q) from block slot L % NB (the block has landed)
    auto load = [&](auto qc, Frag<D> &F, int L) {
        constexpr int Q = decltype(qc)::value;
        const uint32_t st = base + (L & (NB - 1)) * C::SLOT + 16 * Q * C::RB;
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
            ldsm_x4(st + C::BLK + offB[kk], F.kB[kk][0], F.kB[kk][1], F.kB[kk][2], F.kB[kk][3]);
            ldsm_x4_t(st + C::BLK + offA[kk], F.kT[kk][0], F.kT[kk][1], F.kT[kk][2], F.kT[kk][3]);
            ldsm_x4(st + offA[kk], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3]);
        }
        ldsm_x4_t(st + 2 * C::BLK + offV, F.vv[0][0], F.vv[0][1], F.vv[1][0], F.vv[1][1]);
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
    __nv_bfloat16 *const zlane = p.z + (size_t)bh * T * D + (size_t)g * D + col0 + 2 * t4;

    // one chunk (L, Q) on fragments F; fetches chunk (L, Q+1) or (L+1, 0) into Fn.
    // FULL: the chunk has 16 tokens (no bounds masks).  Returns false when there
    // is no next chunk (or a wait gave up).
    auto chunk = [&](auto qc, auto fullc, Frag<D> &F, Frag<D> &Fn, int L) -> bool {
        constexpr int Q = decltype(qc)::value;
        constexpr bool FULL = decltype(fullc)::value;
        const int t0 = 64 * L + 16 * Q;
        const int c = FULL ? 16 : T - t0;
        float e[2][2][4] = {}, sc[2][4] = {}, zc[2][4] = {};
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {  // E^T = W^T K^T
            mma_bf16(e[kk & 1][0], wb[4 * kk], wb[4 * kk + 1], wb[4 * kk + 2], wb[4 * kk + 3], F.kB[kk][0],
                     F.kB[kk][1]);
            mma_bf16(e[kk & 1][1], wb[4 * kk], wb[4 * kk + 1], wb[4 * kk + 2], wb[4 * kk + 3], F.kB[kk][2],
                     F.kB[kk][3]);
        }
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {  // S = Q K^T (off the serial chain)
            mma_bf16(sc[0], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3], F.kB[kk][0], F.kB[kk][1]);
            mma_bf16(sc[1], F.qa[kk][0], F.qa[kk][1], F.qa[kk][2], F.qa[kk][3], F.kB[kk][2], F.kB[kk][3]);
        }
        // next chunk's fragments: inside a block the load is unconditional (reads of
        // the ring past the sequence end stay in bounds and are never used), so the
        // chunk body stays one basic block; crossing into the next block waits for it
        const bool more = t0 + 16 < T;
        if constexpr (Q < 3) {
            load(std::integral_constant<int, Q + 1>{}, Fn, L);
        } else if (more) {
            __syncwarp();
            if (lane == 0) mbar_arrive(blk_empty + 8 * (L & (NB - 1)));
            if (!mbar_wait(blk_full + 8 * ((L + 1) & (NB - 1)), ((L + 1) / NB) & 1, p.status,
                           kSiteConsumerFull))
                return false;
            load(std::integral_constant<int, 0>{}, Fn, L + 1);
        }
        // -Et^T as an A fragment
        float ne[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t vw = F.vv[nt][i >> 1];
                const float vval = (i & 1) ? bf16_hi(vw) : bf16_lo(vw);
                const float r = e[0][nt][i] + e[1][nt][i] - vval;
                ne[nt][i] = (FULL || (8 * nt + 2 * t4 + (i & 1)) < c) ? -F.et[nt][i & 1] * r : 0.f;
            }
        const uint32_t ea0 = pack_bf16(ne[0][0], ne[0][1]), ea1 = pack_bf16(ne[0][2], ne[0][3]);
        const uint32_t ea2 = pack_bf16(ne[1][0], ne[1][1]), ea3 = pack_bf16(ne[1][2], ne[1][3]);
#pragma unroll
        for (int j2 = 0; j2 < NK; ++j2) {  // W^T += (-Et^T) K
            mma_bf16(wacc[2 * j2], ea0, ea1, ea2, ea3, F.kT[j2][0], F.kT[j2][1]);
            mma_bf16(wacc[2 * j2 + 1], ea0, ea1, ea2, ea3, F.kT[j2][2], F.kT[j2][3]);
        }
        // Z = Q W + (mask .* S)(-Et), masked scores as an A fragment from registers
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
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
        convert();
        __nv_bfloat16 *zb = zlane + (size_t)t0 * D;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            if (FULL || g < c)
                *reinterpret_cast<uint32_t *>(zb + 8 * hh) = pack_bf16(zc[hh][0], zc[hh][1]);
            if (FULL || g + 8 < c)
                *reinterpret_cast<uint32_t *>(zb + 8 * D + 8 * hh) = pack_bf16(zc[hh][2], zc[hh][3]);
        }
        return more;
    };
    auto step = [&](auto qc, Frag<D> &F, Frag<D> &Fn, int L) -> bool {
        if (64 * L + 16 * decltype(qc)::value + 16 <= T)
            return chunk(qc, std::true_type{}, F, Fn, L);
        return chunk(qc, std::false_type{}, F, Fn, L);
    };

    if (nblk > 0 && mbar_wait(blk_full, 0, p.status, kSiteConsumerFull)) {
        Frag<D> FA, FB;
        load(std::integral_constant<int, 0>{}, FA, 0);
        for (int L = 0;; ++L) {  // two fragment sets alternate: no register copies
            if (!step(std::integral_constant<int, 0>{}, FA, FB, L)) break;
            if (!step(std::integral_constant<int, 1>{}, FB, FA, L)) break;
            if (!step(std::integral_constant<int, 2>{}, FA, FB, L)) break;
            if (!step(std::integral_constant<int, 3>{}, FB, FA, L)) break;
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
int launch_b16_t(const LinearArgs &a)
{
    using C = B16Cfg<D>;
    CUtensorMap maps[3];
    if (!encode_qkv(maps, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 64)) return -4;
    auto kern = ttt_linear_b16_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return -4;
    B16Params p;
    p.H = a.H;
    p.T = a.T;
    p.causal = a.causal;
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

}  // namespace

int launch_linear_b16(const LinearArgs &a)
{
    switch (a.d) {
    case 16: return launch_b16_t<16>(a);
    case 32: return launch_b16_t<32>(a);
    case 64: return launch_b16_t<64>(a);
    default: return launch_linear_bf16(a);
    }
}

}  // namespace ttt
