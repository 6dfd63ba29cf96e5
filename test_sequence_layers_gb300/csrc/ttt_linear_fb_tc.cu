// ttt_linear_fb_tc.cu -- TTT-Linear forward for one full-batch mini-batch (b >= T,
// non-causal, one inner epoch) on the 5th-generation tensor cores: bf16 operands in
// shared memory, fp32 accumulators in tensor memory, d = 64, T <= 256.
//
// The full-batch step ("ViT3" article, observations 2-3: one inner GD step over all N
// tokens, every query reading the updated weights; "Learning to (Learn at Test Time)",
// section 1.2.2, the mini-batch rule with b = N) is three dense products per
// (batch, head):
//
//   E = K W0 - V            (tokens x d, contraction over the d features)
//   W1^T = W0^T + Et^T K    (d x d, contraction over the tokens; Et = -diag(eta) E)
//   Z = Q W1                (tokens x d)
//
// (negative dot-product loss: E = -V, no first product).  One CTA per (batch, head),
// three per SM (73 KB of shared memory, 128 tensor-memory columns), four warps:
//  * K and V land by TMA in 64-token boxes with the 128-byte swizzle, which is the
//    K-major operand layout of the tensor core for rows of 64 bf16; the K tile is at
//    the same time the MN-major operand (tokens as the reduction dimension) of the
//    update, after which Q takes its place;
//  * one thread issues the tcgen05 products (M = 128 tokens per tile for E and Z,
//    M = 64 for the update) and commits them to an mbarrier;
//  * each thread owns one token row of a tile in the epilogues: it reads its row of
//    E from tensor memory, forms -eta (E - V) and writes it over its own row of V,
//    which is then the MN-major A operand of the update; after the update the first
//    16 lanes of each warp own one column of W1, add W0, write W_out and the bf16
//    W1^T tile of the last product; the Z rows go from tensor memory to global memory.
#include <cuda.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"
#include "ttt_tcgen05.cuh"

namespace ttt {
namespace {

struct FbtCfg {
    static constexpr int D = 64, THREADS = 128;
    static constexpr int TILE = 128 * 128;               // 128 token rows of 128 bytes
    static constexpr int K_OFF = 0, V_OFF = 2 * TILE;    // 2 tiles each; Q replaces K
    static constexpr int W_OFF = 4 * TILE;               // W0^T, then W1^T: 64 rows of 128 bytes
    static constexpr int BAR_OFF = W_OFF + 64 * 128;     // kv, q, mma barriers, one barrier nothing
                                                         // arrives at (timeout test), TMEM address
    static constexpr int SMEM = BAR_OFF + 40 + 1024;
    static constexpr int TMEM_COLS = 128;                // E, then the update, then Z: 2 x 64 columns
};

struct FbtParams {
    int H, T, dot;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    __nv_bfloat16 *z;
    float *W_out;
    int *status;
    unsigned long long test_stall_ns;  // > 0: the timeout test (first wait on a dead barrier)
};

__global__ void __launch_bounds__(FbtCfg::THREADS, 3)
    ttt_linear_fb_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                            const __grid_constant__ CUtensorMap tv, const FbtParams p)
{
    using C = FbtCfg;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gb = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, T = p.T;
    const int ntile = T > 128 ? 2 : 1, nbox = 2 * ntile, nk = (T + 15) >> 4;
    const uint32_t sK = base + C::K_OFF, sV = base + C::V_OFF, sQ = sK, sW = base + C::W_OFF;
    const uint32_t bar_kv = base + C::BAR_OFF, bar_q = bar_kv + 8, bar_mma = bar_kv + 16, dead = bar_kv + 24;
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gb + C::BAR_OFF + 32);

    if (tid == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        mbar_init(bar_kv, 1);
        mbar_init(bar_q, 1);
        mbar_init(bar_mma, 1);
        mbar_init(dead, 1);
        fence_barrier_init();
        // every box of the tiles in use (rows past T arrive as zeros)
        mbar_arrive_expect_tx(bar_kv, 2 * nbox * 8192);
        for (int L = 0; L < nbox; ++L) {
            tma_load_3d(sK + L * 8192, &tk, bar_kv, 0, 64 * L, bh);
            tma_load_3d(sV + L * 8192, &tv, bar_kv, 0, 64 * L, bh);
        }
    }
    if (warp == 0) tc_alloc(base + C::BAR_OFF + 32, C::TMEM_COLS);
    // Lanes 0..15 of warp q own column j = 16 q + lane of W: they read W0's column j
    // (kept for the update's epilogue) and write it as row j of the bf16 W0^T tile, the
    // B operand of E = K W0
    const float *W0 = p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * D * D;
    const int j = 16 * warp + (lane & 15);
    float w0c[D];
#pragma unroll
    for (int i = 0; i < D; ++i) w0c[i] = W0[(size_t)i * D + j];
    if (lane < 16)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4 *>(gb + C::W_OFF + j * 128 + (((uint32_t)ch ^ (uint32_t)(j & 7)) << 4)) =
                make_uint4(pack_bf16(w0c[8 * ch], w0c[8 * ch + 1]), pack_bf16(w0c[8 * ch + 2], w0c[8 * ch + 3]),
                           pack_bf16(w0c[8 * ch + 4], w0c[8 * ch + 5]), pack_bf16(w0c[8 * ch + 6], w0c[8 * ch + 7]));
    fence_proxy_async();  // the generic-proxy writes of W0^T before the tensor core reads them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;

    // ---------------------------------------------------------------- E = K W0
    // the timeout test: the first wait is on a barrier nothing arrives at, and every
    // thread then leaves the products (the copies are still drained below)
    const bool stalled = p.test_stall_ns != 0 && !mbar_wait(dead, 0, p.status, kSiteConsumerFull, p.test_stall_ns);
    if (tid == 0) {
        if (!p.dot && !stalled && mbar_wait(bar_kv, 0, p.status, kSiteConsumerFull)) {
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
            for (int m = 0; m < ntile; ++m)
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma(tmem + 64 * m, sdesc(sK + m * C::TILE + 32 * kk, 16), sdesc(sW + 32 * kk, 16), id, kk > 0);
        }
        tc_commit(bar_mma);  // (arrives at once when no product was issued)
    }
    ok = !stalled && mbar_wait(bar_kv, 0, p.status, kSiteConsumerFull) &&
         mbar_wait(bar_mma, 0, p.status, kSiteConsumerReady);
    tc_fence_after();

    // Et rows: -eta_t (E - V) over this thread's rows of V (zero past T)
    if (ok) {
        for (int m = 0; m < ntile; ++m) {
            if (128 * m + 32 * warp >= 16 * nk) break;  // rows the update does not read (warp-uniform)
            const int t = 128 * m + 32 * warp + lane;
            const float et = t < T ? (p.eta ? p.eta[(size_t)bh * T + t] : p.eta_scalar) : 0.f;
            uint8_t *vrow = gb + C::V_OFF + t * 128;
            float e[64];
            if (!p.dot) tc_ld64(tmem + ((uint32_t)(32 * warp) << 16) + 64 * m, e);
            else
#pragma unroll
                for (int i = 0; i < 64; ++i) e[i] = 0.f;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {  // 16-byte chunks of 8 columns
                uint4 *pc = reinterpret_cast<uint4 *>(vrow + (((uint32_t)ch ^ (uint32_t)(t & 7)) << 4));
                const uint4 vv = *pc;
                const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
                uint32_t ow[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float r0 = e[8 * ch + 2 * q] - bf16_lo(vw[q]);
                    const float r1 = e[8 * ch + 2 * q + 1] - bf16_hi(vw[q]);
                    ow[q] = pack_bf16(-et * r0, -et * r1);
                }
                *pc = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
        }
    }
    fence_proxy_async();  // Et rows before the tensor core reads them
    tc_fence_before();
    ok = __syncthreads_and(ok);
    tc_fence_after();

    // ------------------------------------------------ update: W1^T - W0^T = Et^T K
    // (E's tensor-memory columns are free: every thread has read its rows)
    if (tid == 0 && ok) {
        constexpr uint32_t id = idesc_bf16(64, 64, true, true);
        for (int kk = 0; kk < nk; ++kk)
            tc_mma(tmem, sdesc(sV + 2048 * kk, 8192), sdesc(sK + 2048 * kk, 8192), id, kk > 0);
        tc_commit(bar_mma);
    }
    // lanes 0..15 of warp q own column j = 16 q + lane of W (TMEM lanes 32q .. 32q+15
    // hold rows 16q .. 16q+15 of an M = 64 product)
    ok = ok && mbar_wait(bar_mma, 1, p.status, kSiteConsumerReady);
    tc_fence_after();
    bool q_issued = false;
    if (tid == 0 && ok) {  // the update has read K: Q takes its place
        q_issued = true;
        fence_proxy_async();
        mbar_arrive_expect_tx(bar_q, nbox * 8192);
        for (int L = 0; L < nbox; ++L) tma_load_3d(sQ + L * 8192, &tq, bar_q, 0, 64 * L, bh);
    }
    if (ok) {
        float w1[64];
        tc_ld64(tmem + ((uint32_t)(32 * warp) << 16), w1);  // (warp-wide)
        if (lane < 16) {
#pragma unroll
            for (int i = 0; i < D; ++i) w1[i] += w0c[i];
            if (p.W_out) {
                float *Wo = p.W_out + (size_t)bh * D * D + j;
#pragma unroll
                for (int i = 0; i < D; ++i) Wo[(size_t)i * D] = w1[i];
            }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)  // W1^T row j
                *reinterpret_cast<uint4 *>(gb + C::W_OFF + j * 128 + (((uint32_t)ch ^ (uint32_t)(j & 7)) << 4)) =
                    make_uint4(pack_bf16(w1[8 * ch], w1[8 * ch + 1]), pack_bf16(w1[8 * ch + 2], w1[8 * ch + 3]),
                               pack_bf16(w1[8 * ch + 4], w1[8 * ch + 5]), pack_bf16(w1[8 * ch + 6], w1[8 * ch + 7]));
        }
    }
    fence_proxy_async();  // W1^T rows before the tensor core reads them
    tc_fence_before();
    ok = __syncthreads_and(ok);
    tc_fence_after();

    // ---------------------------------------------------------------- Z = Q W1
    if (tid == 0 && ok) {
        if (mbar_wait(bar_q, 0, p.status, kSiteConsumerFull)) {
            constexpr uint32_t id = idesc_bf16(128, 64, false, false);
            for (int m = 0; m < ntile; ++m)
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma(tmem + 64 * m, sdesc(sQ + m * C::TILE + 32 * kk, 16), sdesc(sW + 32 * kk, 16), id, kk > 0);
        }
        tc_commit(bar_mma);
    }
    ok = ok && mbar_wait(bar_q, 0, p.status, kSiteConsumerFull) && mbar_wait(bar_mma, 0, p.status, kSiteConsumerReady);
    tc_fence_after();
    if (ok) {
        for (int m = 0; m < ntile; ++m) {
            if (128 * m + 32 * warp >= T) break;  // no token of this warp's rows (warp-uniform)
            const int t = 128 * m + 32 * warp + lane;
            __nv_bfloat16 *zr = p.z + ((size_t)bh * T + t) * D;
            float zz[64];
            tc_ld64(tmem + ((uint32_t)(32 * warp) << 16) + 64 * m, zz);  // (warp-wide)
            if (t < T) {
                uint4 *dst = reinterpret_cast<uint4 *>(zr);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    dst[ch] = make_uint4(pack_bf16(zz[8 * ch], zz[8 * ch + 1]), pack_bf16(zz[8 * ch + 2], zz[8 * ch + 3]),
                                         pack_bf16(zz[8 * ch + 4], zz[8 * ch + 5]),
                                         pack_bf16(zz[8 * ch + 6], zz[8 * ch + 7]));
            }
        }
    }
    // copies still landing (after a timeout) end before the CTA does
    if (tid == 0) {
        mbar_wait(bar_kv, 0, p.status, kSiteDrain);
        if (q_issued) mbar_wait(bar_q, 0, p.status, kSiteDrain);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tc_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace

// b >= T (one mini-batch), non-causal, one epoch, no inner norm, d = 64, bf16, T <= 256;
// -2 otherwise.
int launch_linear_fb_tc(const LinearArgs &a)
{
    using C = FbtCfg;
    if (a.d != 64 || a.causal || a.b < a.T || a.T > 256 || a.T < 1 || a.epochs != 1 || a.ln_gamma) return -2;
    CUtensorMap maps[3];
    if (!encode_qkv(maps, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 64)) return -4;
    if (cudaFuncSetAttribute(ttt_linear_fb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
        return -4;
    FbtParams p;
    p.H = a.H;
    p.T = a.T;
    p.dot = a.loss;
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W0 = a.W0;
    p.w0_bstride = a.w0_bstride;
    p.z = static_cast<__nv_bfloat16 *>(a.z);
    p.W_out = a.W_out;
    p.status = a.status;
    p.test_stall_ns = a.test_stall_ns;
    ttt_linear_fb_tc_kernel<<<a.B * a.H, C::THREADS, C::SMEM, a.stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace ttt
