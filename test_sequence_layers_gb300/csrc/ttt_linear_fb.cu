// ttt_linear_fb.cu -- TTT-Linear forward for one full-batch mini-batch (b = T,
// non-causal), bf16 operands, fp32 accumulation and state, d = 64, T <= 256.
//
// The full-batch variant ("ViT3" article, observations 2-3: one inner GD step over
// all N tokens, every query reads the updated weights; "Learning to (Learn at Test
// Time)", section 1.2.2 for the mini-batch rule with b = N) has no serial chain:
// every token's residual is taken at the start weights W0, so
//
//   E = K W0 - V,   W1 = W0 - K^T diag(eta) E,   Z = Q W1
//
// With several inner epochs (the same article, observation 2: one epoch of
// full-batch inner training is one update over all N tokens) the E / update pass
// repeats from the W the previous pass left while K and V are still on chip; with
// the negative dot-product loss the residual is -V.
//
// are three independent passes over 16-token chunks.  One CTA per (batch, head):
// the whole sequence's K and V land in shared memory with one TMA load per 64-token
// box (one mbarrier per box, so the update pass starts on the first), Q replaces V
// once the update pass is done, and four warps (16 output columns each, W^T as fp32
// mma accumulators, as in the mini-batch kernels) run the E / update pass and the
// Z pass.  Three CTAs fit on an SM, so one CTA's loads overlap the others' products.
#include <cuda.h>

#include <type_traits>

#include "ttt_device.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

struct FbCfg {
    static constexpr int D = 64, NCW = 4, THREADS = NCW * 32;
    static constexpr int NJ = D / 8, NK = D / 16;
    static constexpr int RB = 2 * D;          // 128 bytes per token row
    static constexpr int BLK = 64 * RB;       // one 64-token box (8 KB)
    static constexpr int MAXT = 256;          // longest sequence held on chip
    // shared memory for a sequence of nblk 64-token boxes: K, V (then Q in V's
    // place), eta, barriers (one per K/V box pair, one for all of Q)
    static constexpr int smem_bytes(int nblk) { return 2 * nblk * BLK + MAXT * 4 + 8 * (MAXT / 64 + 1) + 1024; }
};

// Offset of element (r, c) inside a run of 64-token boxes written by TMA with the
// 128-byte swizzle; rows of consecutive boxes follow each other.
__device__ __forceinline__ uint32_t fboff(int r, int c)
{
    const uint32_t a = static_cast<uint32_t>(r * FbCfg::RB + c * 2);
    return a ^ (((a >> 7) & 7u) << 4);
}

struct FbParams {
    int H, T, dot, epochs;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    __nv_bfloat16 *z;
    float *W_out;
    int *status;
};

__global__ void __launch_bounds__(FbCfg::THREADS, 3)
    ttt_linear_fb_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, const FbParams p)
{
    using C = FbCfg;
    constexpr int D = C::D, NJ = C::NJ, NK = C::NK;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x, T = p.T;
    const int nblk = (T + 63) >> 6, nch = (T + 15) >> 4;
    const uint32_t sK = base, sV = base + nblk * C::BLK, sQ = sV;  // Q replaces V after the update pass
    float *eta_s = reinterpret_cast<float *>(gbase + 2 * nblk * C::BLK);
    const uint32_t kv_bar = base + 2 * nblk * C::BLK + C::MAXT * 4;  // [nblk] K, V of box L landed
    const uint32_t q_bar = kv_bar + 8 * nblk;                          // all of Q landed
    const bool has_eta = p.eta != nullptr;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        for (int L = 0; L <= nblk; ++L) mbar_init(kv_bar + 8 * L, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && nblk > 0) {  // K, V box by box (the update pass starts on the first)
        for (int L = 0; L < nblk; ++L) {
            mbar_arrive_expect_tx(kv_bar + 8 * L, 2 * C::BLK);
            tma_load_3d(sK + L * C::BLK, &tk, kv_bar + 8 * L, 0, 64 * L, bh);
            tma_load_3d(sV + L * C::BLK, &tv, kv_bar + 8 * L, 0, 64 * L, bh);
        }
    }
    for (int i = threadIdx.x; i < T; i += C::THREADS) eta_s[i] = has_eta ? p.eta[(size_t)bh * T + i] : p.eta_scalar;

    // W^T[col0+g (+8)][8j+2t4 .. +1] of this warp's 16 output columns
    const int w = warp, col0 = 16 * w, g = lane >> 2, t4 = lane & 3;
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
    // bf16 W as the A operand of E^T = W^T K^T (k-tile kk: words 4kk .. 4kk+3) and
    // as the B operand of Z = Q W
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
    const int rowA = (lane & 7) + 8 * ((lane >> 3) & 1), colA = 8 * (lane >> 4);
    const int rowB = (lane & 7) + 8 * (lane >> 4), colB = 8 * ((lane >> 3) & 1);
    // per-lane fragment offsets inside a 16-token chunk; a chunk starting at token
    // t0 (a multiple of 16) adds t0 * 128 bytes (the swizzle key is the row mod 8)
    uint32_t offA[NK], offB[NK];
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
        offA[kk] = fboff(rowA, 16 * kk + colA);
        offB[kk] = fboff(rowB, 16 * kk + colB);
    }
    const uint32_t offV = fboff(rowB, col0 + colB);
    __syncthreads();  // eta staged
    bool ok = true;

    // one 16-token chunk of the E / update pass (the residuals all read W0 = wb,
    // the writes accumulate in wacc); FULL: no token of the chunk is past T
    auto upd_chunk = [&](auto fullc, int t0) {
        constexpr bool FULL = decltype(fullc)::value;
        const uint32_t ck = sK + t0 * C::RB;
        float e[2][2][4] = {};
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {  // E^T = W^T K^T (no product for the dot loss)
            if (p.dot) break;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ck + offB[kk], b0, b1, b2, b3);
            mma_bf16(e[kk & 1][0], wb[4 * kk], wb[4 * kk + 1], wb[4 * kk + 2], wb[4 * kk + 3], b0, b1);
            mma_bf16(e[kk & 1][1], wb[4 * kk], wb[4 * kk + 1], wb[4 * kk + 2], wb[4 * kk + 3], b2, b3);
        }
        uint32_t vv[2][2];
        ldsm_x4_t(sV + t0 * C::RB + offV, vv[0][0], vv[0][1], vv[1][0], vv[1][1]);
        const float2 et0 = *reinterpret_cast<const float2 *>(eta_s + t0 + 2 * t4);
        const float2 et1 = *reinterpret_cast<const float2 *>(eta_s + t0 + 8 + 2 * t4);
        const float et[2][2] = {{et0.x, et0.y}, {et1.x, et1.y}};
        float ne[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t vw = vv[nt][i >> 1];
                const float vval = (i & 1) ? bf16_hi(vw) : bf16_lo(vw);
                const float r = e[0][nt][i] + e[1][nt][i] - vval;
                ne[nt][i] = (FULL || t0 + 8 * nt + 2 * t4 + (i & 1) < T) ? -et[nt][i & 1] * r : 0.f;
            }
        const uint32_t ea0 = pack_bf16(ne[0][0], ne[0][1]), ea1 = pack_bf16(ne[0][2], ne[0][3]);
        const uint32_t ea2 = pack_bf16(ne[1][0], ne[1][1]), ea3 = pack_bf16(ne[1][2], ne[1][3]);
#pragma unroll
        for (int j2 = 0; j2 < NK; ++j2) {  // W^T += (-Et^T) K
            uint32_t k0, k1, k2, k3;
            ldsm_x4_t(ck + offA[j2], k0, k1, k2, k3);
            mma_bf16(wacc[2 * j2], ea0, ea1, ea2, ea3, k0, k1);
            mma_bf16(wacc[2 * j2 + 1], ea0, ea1, ea2, ea3, k2, k3);
        }
    };
    for (int ep = 0; ep < p.epochs && ok; ++ep) {
        for (int c = 0; c < nch && ok; ++c) {
            if (ep == 0 && (c & 3) == 0) ok = mbar_wait(kv_bar + 8 * (c >> 2), 0, p.status, kSiteConsumerFull);
            if (16 * c + 16 <= T) upd_chunk(std::true_type{}, 16 * c);
            else upd_chunk(std::false_type{}, 16 * c);
        }
        convert();  // the next pass's residuals (and finally Z) read these weights
    }
    // Q into V's place once no warp reads V any more
    __syncthreads();
    if (threadIdx.x == 0 && nblk > 0 && ok) {
        fence_proxy_async();
        mbar_arrive_expect_tx(q_bar, nblk * C::BLK);
        for (int L = 0; L < nblk; ++L) tma_load_3d(sQ + L * C::BLK, &tq, q_bar, 0, 64 * L, bh);
    }
    ok = __syncthreads_and(ok) && (nblk == 0 || mbar_wait(q_bar, 0, p.status, kSiteConsumerFull));
    if (ok) {
        // Z pass: every query reads W1
        __nv_bfloat16 *zlane = p.z + (size_t)bh * T * D + (size_t)g * D + col0 + 2 * t4;
#pragma unroll 2
        for (int c = 0; c < nch; ++c) {
            const int t0 = 16 * c;
            float zc[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(sQ + t0 * C::RB + offA[kk], a0, a1, a2, a3);
                mma_bf16(zc[0], a0, a1, a2, a3, wb[4 * kk], wb[4 * kk + 2]);
                mma_bf16(zc[1], a0, a1, a2, a3, wb[4 * kk + 1], wb[4 * kk + 3]);
            }
            __nv_bfloat16 *zb = zlane + (size_t)t0 * D;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (t0 + g < T) *reinterpret_cast<uint32_t *>(zb + 8 * hh) = pack_bf16(zc[hh][0], zc[hh][1]);
                if (t0 + g + 8 < T)
                    *reinterpret_cast<uint32_t *>(zb + 8 * D + 8 * hh) = pack_bf16(zc[hh][2], zc[hh][3]);
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

}  // namespace

// b >= T (one mini-batch), non-causal, d = 64, bf16, T <= 256; -2 otherwise.
int launch_linear_fb(const LinearArgs &a)
{
    using C = FbCfg;
    if (a.d != 64 || a.causal || a.b < a.T || a.T > C::MAXT) return -2;
    CUtensorMap maps[3];
    if (!encode_qkv(maps, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 64)) return -4;
    const int smem = C::smem_bytes((a.T + 63) / 64);
    if (cudaFuncSetAttribute(ttt_linear_fb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return -4;
    FbParams p;
    p.H = a.H;
    p.T = a.T;
    p.dot = a.loss;
    p.epochs = a.epochs;
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W0 = a.W0;
    p.w0_bstride = a.w0_bstride;
    p.z = static_cast<__nv_bfloat16 *>(a.z);
    p.W_out = a.W_out;
    p.status = a.status;
    ttt_linear_fb_kernel<<<a.B * a.H, C::THREADS, smem, a.stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace ttt
