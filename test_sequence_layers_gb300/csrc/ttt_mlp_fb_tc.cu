// ttt_mlp_fb_tc.cu -- TTT-MLP forward for one full-batch mini-batch (b >= T,
// non-causal, one inner step) on the 5th-generation tensor cores: d = 64, hidden
// width m = 256, bf16 tokens, fp32 inner weights, any T >= 1.
//
// The full-batch step ("ViT3" article, observations 2 and 4: one inner GD step over
// all N tokens with a SiLU MLP of width ratio 4, every query reading the updated
// weights; "Learning to (Learn at Test Time)" walkthrough, section 2.2.1, the
// two-layer inner model) takes every gradient at the start weights:
//
//   H  = K W1 + c1,  A = act(H)                  (tokens x m)
//   Et = -diag(eta) (A W2 + c2 - V)              (tokens x d)
//   Dl = (Et W2^T) .* act'(H)                    (tokens x m)
//   W1 += K^T Dl, c1 += 1^T Dl, W2 += A^T Et, c2 += 1^T Et
//   Z  = act(Q W1 + c1) W2 + c2                  (updated weights)
//
// One persistent CTA per SM works through (batch, head) chains.  Nine warps:
//  * warp 8 (one thread) issues the TMA loads of K/V (then Q) tiles into a
//    two-stage ring and every tcgen05 product, and commits them to mbarriers;
//  * warps 0-7 do the elementwise work from tensor memory: warp w reads TMEM lanes
//    32 (w % 4) .. +31 and columns half w / 4 of each 64-column chunk.
// A warp can only reach its own quarter of the 128 TMEM lanes, so a tile's rows are
// dealt out evenly: with nt = ceil(T / 128) tiles, each 32-row quarter of a tile
// holds R = ceil(T / (4 nt)) consecutive tokens (a 32-row TMA box at token
// R (4 tile + quarter)); its rows R .. 31 repeat the next tokens or read zeros past
// T, and take eta = 0, so they add nothing to the weight writes.
// Products, operands in 128-byte-swizzled shared memory (K-major: rows of 64
// bf16 along the reduction; MN-major: the same rows read across):
//  * token side, M = 128 rows, N = 64: H chunk c (hidden 64c .. 64c+63) = K W1,
//    E = sum_c A_c W2_c, P chunk c = Et W2^T, and in the output pass H_q, Z;
//  * weight side, M = 128 hidden units, contracted over the tile's rows:
//    W2 += A^T Et (N = 64) and [W1^T | c1] += Dl^T [K | 1] (N = 80: a tile of ones
//    is the second 64-feature atom of B, so the c1 write comes with W1's),
//    accumulated in tensor memory that starts out holding the chain's start
//    weights (fp32);
//  * the c2 write Et^T 1 (M = 64 features, N = 16) against the ones tile.
// H / P chunks alternate between two 64-column tensor-memory slots, so the
// elementwise work on one chunk overlaps the product of the next.  Activations A
// (later Dl, and A_q in the output pass) are written as bf16 into a [128][256]
// tile that is at once the K-major operand of the token-side products and the
// MN-major operand of the weight side; act'(H) stays in registers as packed bf16.
// At the end of the update pass thread h owns hidden unit h: it writes the bf16
// copies of its rows of the updated W1^T and W2 that the output pass reads, and
// the final c1, c2; the fp32 rows of W1 and W2 leave one batch per chunk during the
// first output tile, and during a chain's last output tile the next chain's start
// weights are loaded, one batch per chunk, into the freed weight accumulators (W2
// rows through a per-warp piece of the idle Et tile, so global memory sees whole
// row pieces).
//
// The LN instantiation carries the inner norm and residual, f(x) = x + LN(y) (the
// walkthrough's TTT-MLP): the E stage forms the norm's backward and the output pass
// z = q + LN(y_q), each token's statistics combined from the two warps of its lane
// quarter at a 64-thread named barrier.
//
// Every wait is bounded; a timeout records its site in the status word, raises a
// CTA-wide abort flag, and all warps unwind: elementwise warps that gave up stop
// arriving on mbarriers but pass every named barrier, the issuing thread leaves at
// its next wait and drains the copies and products it issued before tensor memory
// is released.
#include <cuda.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"
#include "ttt_tcgen05.cuh"

namespace ttt {
namespace {

struct FmtCfg {
    static constexpr int D = 64, M = 256;
    static constexpr int NCW = 8;                        // elementwise warps
    static constexpr int THREADS = (NCW + 1) * 32;       // + the issuing warp
    static constexpr int TILE = 128 * 128;               // 128 rows of 64 bf16
    static constexpr int BOX = 32 * 128;                 // one quarter: 32 rows
    static constexpr int STAGE = 2 * TILE;               // K (or Q), V
    static constexpr int W1_OFF = 2 * STAGE;             // bf16 W1^T [256 hidden][64]
    static constexpr int W2_OFF = W1_OFF + 2 * TILE;     // bf16 W2 [256 hidden][64]
    static constexpr int A_OFF = W2_OFF + 2 * TILE;      // bf16 A / Dl / A_q: 4 x [128 rows][64 hidden]
    static constexpr int ET_OFF = A_OFF + 4 * TILE;      // bf16 Et [128 rows][64]
    static constexpr int ONES_OFF = ET_OFF + TILE;       // bf16 ones [128][64]
    static constexpr int F_OFF = ONES_OFF + TILE;        // fp32 c1[256], c2[64]
    static constexpr int LN_OFF = F_OFF + 4 * (M + D);   // fp32 inner-norm gamma[64], beta[64]
    static constexpr int BAR_OFF = LN_OFF + 4 * 2 * D;
    static constexpr int NBAR = 17;
    static constexpr int SMEM = BAR_OFF + NBAR * 8 + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    // tensor-memory columns: chunk slots, E / Z, [W1^T | c1] (two 128-row tiles of 64 + 16
    // columns, the c1 entry in the first of the 16), W2 (two tiles), c2 writes (an M = 64
    // product)
    static constexpr uint32_t T_SLOT = 0, T_E = 128, T_W1 = 192, W1C = 80, T_W2 = 352, T_C2 = 480;
};
static_assert(FmtCfg::SMEM <= 227 * 1024, "shared memory");

// barrier indices
enum : int {
    B_FULL = 0,      // [2] a token tile landed (TMA)
    B_SFULL = 2,     // [2] an H / P chunk is in its slot (commit)
    B_SFREE = 4,     // [2] the slot was read and its bf16 chunk written (8 warps)
    B_EFULL = 6,     // E or Z accumulated (commit)
    B_ETREADY = 7,   // Et written (8 warps)
    B_AFREE = 8,     // [2] the W2 write has read A of hidden units 128 i .. (commit)
    B_WDONE = 10,    // every product of the update pass is done (commit)
    B_WREADY = 11,   // updated bf16 weights and biases in place (8 warps)
    B_WSTART = 12,   // a chain's start weights in place (8 warps)
    B_STFREE = 13,   // [2] the products have read a stage (commit)
    B_DRAIN = 15,    // end of the issuer's products (commit)
    B_DEAD = 16,     // nothing arrives here (the timeout test)
};

struct FmtParams {
    int BH, H, T, per_batch;
    const float *eta;
    float eta_scalar;
    const float *W1, *c1, *W2, *c2;
    __nv_bfloat16 *z;
    float *W1o, *c1o, *W2o, *c2o;
    int *status;
    const float *ln_gamma, *ln_beta;  // inner norm [H][d] (the LN instantiation)
    float ln_eps;
    const __nv_bfloat16 *q;           // the queries, for the residual z = q + LN(y)
    unsigned long long test_stall_ns;  // > 0: the elementwise warps' first wait is on a dead barrier
};

// GELU(h) = h Phi(h) with Phi the standard normal CDF (ACT 1, norm_cdf), and its
// derivative GELU' = Phi + h phi(h); SiLU (ACT 0) takes the paired path below.
__device__ __forceinline__ float gelu_v(float h)
{
    float e;
    return h * norm_cdf(h, e);
}
__device__ __forceinline__ void gelu_vd(float h, float &a, float &ad)
{
    float e;
    const float Phi = norm_cdf(h, e);
    a = h * Phi;
    ad = fmaf(h * 0.39894228040143268f, e, Phi);
}

// tanh of two values (hardware approximation)
__device__ __forceinline__ float2 tanh2(float2 x)
{
    float2 t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t.x) : "f"(x.x));
    asm("tanh.approx.f32 %0, %1;" : "=f"(t.y) : "f"(x.y));
    return t;
}

// SiLU(h) = h sigma(h) (ViT3 article, observation 4) and SiLU' = sigma + a (1 - sigma),
// two values at a time with paired fp32 arithmetic, sigma = (1 + tanh(h / 2)) / 2 (one
// special-function op per value instead of an exponential and a reciprocal)
__device__ __forceinline__ void silu_d2(float2 h, float2 &a, float2 &ad)
{
    const float2 half2 = make_float2(0.5f, 0.5f), one2 = make_float2(1.f, 1.f), mone2 = make_float2(-1.f, -1.f);
    const float2 t = tanh2(__fmul2_rn(h, half2));
    const float2 s = __ffma2_rn(t, half2, half2);
    a = __fmul2_rn(h, s);
    ad = __ffma2_rn(a, __ffma2_rn(s, mone2, one2), s);  // s + a (1 - s)
}
__device__ __forceinline__ float2 silu2(float2 h)
{
    const float2 half2 = make_float2(0.5f, 0.5f);
    const float2 t = tanh2(__fmul2_rn(h, half2));
    return __fmul2_rn(h, __ffma2_rn(t, half2, half2));
}
__device__ __forceinline__ uint32_t pack2(float2 v) { return pack_bf16(v.x, v.y); }
__device__ __forceinline__ float2 unpack2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ float2 f2(uint32_t lo, uint32_t hi) { return make_float2(__uint_as_float(lo), __uint_as_float(hi)); }

// Waits for a phase; gives up (false) once the CTA's abort flag is up, or after the
// limit, recording `site` and raising the flag.
__device__ __forceinline__ bool fwait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *status,
                                      int site)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                atomicCAS(status, 0, site);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// As fwait, for threads with nothing else to do: each probe may suspend the thread
// (up to a few microseconds) until the phase completes, leaving issue slots to the
// issuing thread.
__device__ __forceinline__ bool fwait_sleep(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *status,
                                            int site, unsigned long long limit_ns = kWaitLimitNs)
{
    const uint64_t t0 = globaltimer();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(4000u)
            : "memory");
        if (done) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            atomicCAS(status, 0, site);
            *abort_flag = 1;
            return false;
        }
    }
}

// byte offset of 16-byte chunk ch of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t swz(int r, int ch)
{
    return (uint32_t)r * 128u + (((uint32_t)ch ^ (uint32_t)(r & 7)) << 4);
}

__device__ __forceinline__ void named_sync_compute() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// the two warps that share a TMEM lane quarter (w and w + 4)
__device__ __forceinline__ void named_sync_pair(int q) { asm volatile("bar.sync %0, 64;" ::"r"(2 + q) : "memory"); }

template <int ACT, bool LN>
__global__ void __launch_bounds__(FmtCfg::THREADS, 1)
    ttt_mlp_fb_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, const FmtParams p)
{
    using C = FmtCfg;
    constexpr int D = C::D, M = C::M;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gb = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T, nt = (T + 127) >> 7, R = (T + 4 * nt - 1) / (4 * nt);
    const uint32_t bars = base + C::BAR_OFF;
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gb + C::BAR_OFF + C::NBAR * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gb + C::BAR_OFF + C::NBAR * 8 + 4);
    float *c1s = reinterpret_cast<float *>(gb + C::F_OFF), *c2s = c1s + M;
    float *gms = reinterpret_cast<float *>(gb + C::LN_OFF), *bts = gms + D;  // inner-norm gamma, beta
    const uint32_t sW1 = base + C::W1_OFF, sW2 = base + C::W2_OFF, sA = base + C::A_OFF, sET = base + C::ET_OFF;
    const uint32_t sONE = base + C::ONES_OFF;
    auto BAR = [&](int i) { return bars + 8u * (uint32_t)i; };

    if (tid == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        for (int i = 0; i < C::NBAR; ++i) {
            const bool eight = i == B_SFREE || i == B_SFREE + 1 || i == B_ETREADY || i == B_WREADY || i == B_WSTART;
            mbar_init(BAR(i), eight ? 8 : 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    for (int i = tid; i < C::TILE / 16; i += C::THREADS)  // the ones tile (bf16 1.0 = 0x3f80)
        *reinterpret_cast<uint4 *>(gb + C::ONES_OFF + 16 * i) =
            make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
    fence_proxy_async();
    if (warp == C::NCW) tc_alloc(base + C::BAR_OFF + C::NBAR * 8, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == C::NCW) {
        // ------------------------------------------------------------ issuer
        if (lane == 0) {
            constexpr uint32_t ID_TOK = idesc_bf16(128, 64, false, false);  // token side, B K-major
            constexpr uint32_t ID_TOKW = idesc_bf16(128, 64, false, true);  // token side, B = W2 read across
            constexpr uint32_t ID_W = idesc_bf16(128, 64, true, true);      // weight side
            constexpr uint32_t ID_W1 = idesc_bf16(128, 80, true, true);     // Dl^T [K | 1]
            constexpr uint32_t ID_C2 = idesc_bf16(64, 16, true, false);     // Et^T 1
            // operand descriptors of the fixed tiles; a byte offset o moves one by o / 16
            const uint64_t dW1 = sdesc(sW1, 16), dW2k = sdesc(sW2, 16), dW2m = sdesc(sW2, 8192);
            const uint64_t dAk = sdesc(sA, 16), dAw = sdesc(sA, C::TILE), dETk = sdesc(sET, 16);
            const uint64_t dETm = sdesc(sET, 8192), dONE = sdesc(sONE, 16);
            // tile g of this CTA: chain g / (2 nt); update tiles, then output tiles
            auto issue_load = [&](int g) -> bool {
                const int ci = g / (2 * nt), rr = g - ci * 2 * nt;
                const int bh = blockIdx.x + ci * gridDim.x;
                if (bh >= p.BH) return false;
                const uint32_t st = base + (uint32_t)(g & 1) * C::STAGE, bar = BAR(B_FULL + (g & 1));
                const int mt = rr < nt ? rr : rr - nt;
                if (rr < nt) {
                    mbar_arrive_expect_tx(bar, 2 * C::TILE);
                    for (int qq = 0; qq < 4; ++qq) {
                        tma_load_3d(st + C::BOX * qq, &tk, bar, 0, R * (4 * mt + qq), bh);
                        tma_load_3d(st + C::TILE + C::BOX * qq, &tv, bar, 0, R * (4 * mt + qq), bh);
                    }
                } else {
                    mbar_arrive_expect_tx(bar, C::TILE);
                    for (int qq = 0; qq < 4; ++qq) tma_load_3d(st + C::BOX * qq, &tq, bar, 0, R * (4 * mt + qq), bh);
                }
                return true;
            };
            int loaded = 0;
            if (issue_load(0)) loaded = 1;
            if (loaded == 1 && issue_load(1)) loaded = 2;
            int g = 0, jj = 0, nu = 0;
            bool ok = true;
            auto wt = [&](int b, uint32_t parity, int site) {
                return ok = ok && fwait(BAR(b), parity, abort_flag, p.status, site);
            };
            // a slot for chunk job jj (waits for job jj - 2 to have been consumed)
            auto slot = [&]() -> uint32_t {
                if (jj >= 2) wt(B_SFREE + (jj & 1), ((jj - 2) >> 1) & 1, kSiteProducerEmpty);
                return tmem + C::T_SLOT + 64u * (uint32_t)(jj & 1);
            };
            auto finish_job = [&]() {
                tc_commit(BAR(B_SFULL + (jj & 1)));
                ++jj;
            };
            // the tile before g has been read by its products: its stage takes tile g + 1
            auto refill = [&]() {
                if (g >= 1 && loaded == g + 1) {
                    if (!wt(B_STFREE + ((g - 1) & 1), ((g - 1) >> 1) & 1, kSiteStage)) return;
                    if (issue_load(g + 1)) ++loaded;
                }
            };
            // chunk c of X W (X = K or Q in stage st, W = the bf16 W1^T tile)
            auto issue_xw = [&](uint32_t st, int c) {
                const uint32_t d = slot();
                if (!ok) return;
                const uint64_t dx = sdesc(st, 16);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc_mma(d, dx + 2 * kk, dW1 + 512 * c + 2 * kk, ID_TOK, kk > 0);
                finish_job();
            };
            auto issue_aw2 = [&](int c) {  // E (or Z) += A_c W2_c
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma(tmem + C::T_E, dAk + 1024 * c + 2 * kk, dW2m + 512 * c + 128 * kk, ID_TOKW, c > 0 || kk > 0);
            };
            for (int ci = 0, bh = blockIdx.x; ok && bh < p.BH; ++ci, bh += gridDim.x) {
                if (!wt(B_WSTART, ci & 1, kSiteConsumerReady)) break;
                tc_fence_after();
                // ------------------------------------------------ update pass
                int jh = 0;  // the current tile's four H chunk jobs are jh .. jh + 3
                for (int mt = 0; mt < nt && ok; ++mt, ++g, ++nu) {
                    const uint32_t sK = base + (uint32_t)(g & 1) * C::STAGE;
                    if (mt == 0) {  // (later tiles' first two chunks go out with the previous tile)
                        if (!wt(B_FULL + (g & 1), (g >> 1) & 1, kSiteConsumerFull)) break;
                        tc_fence_after();
                        jh = jj;
                        issue_xw(sK, 0);
                        issue_xw(sK, 1);
                    }
                    for (int c = 0; c < 4 && ok; ++c) {
                        if (!wt(B_SFREE + ((jh + c) & 1), ((jh + c) >> 1) & 1, kSiteConsumerReady)) break;
                        tc_fence_after();
                        if (c + 2 < 4) issue_xw(sK, c + 2);
                        if (!ok) break;
                        issue_aw2(c);
                    }
                    if (!ok) break;
                    tc_commit(BAR(B_EFULL));
                    refill();  // (here, not at the tile's start: the previous tile's last products are done by now)
                    if (!wt(B_ETREADY, nu & 1, kSiteConsumerReady)) break;
                    tc_fence_after();
                    const int jp = jj;  // the tile's four chunk jobs are jp .. jp + 3
                    auto issue_p = [&](int c) {  // P chunk c = Et W2[64c .., :]^T
                        const uint32_t d = slot();
                        if (!ok) return;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) tc_mma(d, dETk + 2 * kk, dW2k + 512 * c + 2 * kk, ID_TOK, kk > 0);
                        finish_job();
                    };
                    auto issue_w2 = [&](int hc) {  // W2 (hidden 128 hc ..) += A^T Et; A half hc is then free
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc_mma(tmem + C::T_W2 + 64 * hc, dAw + 2048 * hc + 128 * kk, dETm + 128 * kk, ID_W, true);
                        tc_commit(BAR(B_AFREE + hc));
                    };
                    auto issue_w1 = [&](int hc) {  // [W1^T | c1] (hidden 128 hc ..) += Dl^T [K | 1]: the
                        const uint64_t da = dAw + 2048 * hc;  // ones tile is the second 64-feature atom of B
                        const uint64_t dk = sdesc(sK, (uint32_t)(C::ONES_OFF - (g & 1) * C::STAGE));
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc_mma(tmem + C::T_W1 + C::W1C * hc, da + 128 * kk, dk + 128 * kk, ID_W1, true);
                    };
                    const uint32_t sKn = base + (uint32_t)((g + 1) & 1) * C::STAGE;
                    // the products in the order the chunks are consumed: P0, the first W2
                    // write, P1; then each chunk's slot goes to the product two chunks on,
                    // the next tile's first two H chunks included
                    issue_p(0);
                    if (!ok) break;
                    issue_w2(0);
                    issue_p(1);
                    for (int c = 0; c < 4 && ok; ++c) {
                        if (!wt(B_SFREE + ((jp + c) & 1), ((jp + c) >> 1) & 1, kSiteConsumerReady)) break;
                        tc_fence_after();
                        if (c == 0) {
                            issue_p(2);
                            if (!ok) break;
                            issue_w2(1);
                        } else if (c == 1) {
                            issue_p(3);
                            if (!ok) break;
                            issue_w1(0);
                        } else if (mt + 1 < nt) {  // the next tile's H chunk c - 2
                            if (c == 2) {
                                if (!wt(B_FULL + ((g + 1) & 1), ((g + 1) >> 1) & 1, kSiteConsumerFull)) break;
                                tc_fence_after();
                                jh = jj;
                            }
                            issue_xw(sKn, c - 2);
                            if (!ok) break;
                        }
                        if (c == 3) {
                            issue_w1(1);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)  // c2 writes: Et^T 1
                                tc_mma(tmem + C::T_C2, dETm + 128 * kk, dONE + 2 * (kk & 3), ID_C2, mt > 0 || kk > 0);
                        }
                    }
                    if (!ok) break;
                    tc_commit(BAR(B_STFREE + (g & 1)));
                }
                if (!ok) break;
                tc_commit(BAR(B_WDONE));
                if (!wt(B_WREADY, ci & 1, kSiteConsumerReady)) break;
                tc_fence_after();
                // ------------------------------------------------ output pass
                for (int mt = 0; mt < nt && ok; ++mt, ++g) {
                    const uint32_t sQ = base + (uint32_t)(g & 1) * C::STAGE;
                    if (!wt(B_FULL + (g & 1), (g >> 1) & 1, kSiteConsumerFull)) break;
                    tc_fence_after();
                    const int jq = jj;  // the tile's four chunk jobs are jq .. jq + 3
                    issue_xw(sQ, 0);
                    issue_xw(sQ, 1);
                    refill();
                    for (int c = 0; c < 4 && ok; ++c) {
                        if (!wt(B_SFREE + ((jq + c) & 1), ((jq + c) >> 1) & 1, kSiteConsumerReady)) break;
                        tc_fence_after();
                        if (c + 2 < 4) issue_xw(sQ, c + 2);
                        if (!ok) break;
                        issue_aw2(c);
                    }
                    if (!ok) break;
                    tc_commit(BAR(B_EFULL));
                    tc_commit(BAR(B_STFREE + (g & 1)));
                }
            }
            // copies still landing (after a timeout) and products still running end
            // before tensor memory and the CTA do
            for (int x = g; x < loaded; ++x) mbar_wait(BAR(B_FULL + (x & 1)), (x >> 1) & 1, p.status, kSiteDrain);
            tc_commit(BAR(B_DRAIN));
            mbar_wait(BAR(B_DRAIN), 0, p.status, kSiteDrain);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ elementwise warps
        const int q = warp & 3, hh = warp >> 2;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);  // this warp's lane quarter
        const int r = 32 * q + lane;                            // row of the tile
        int jj = 0, ne = 0, nu = 0, g = 0;
        bool ok = true;
        auto wt = [&](int b, uint32_t parity, int site) {
            const bool mine = ok && fwait_sleep(BAR(b), parity, abort_flag, p.status, site);
            ok = __all_sync(0xffffffffu, mine);
            return ok;
        };
        // this warp's shared-memory writes and TMEM reads are done; a warp whose waits
        // gave up stops arriving, so the issuing thread meets the abort flag at once
        auto release = [&](int b) {
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(BAR(b));
        };
        if (p.test_stall_ns)  // the timeout test: a first wait that can only run out
            ok = __all_sync(0xffffffffu, fwait_sleep(BAR(B_DEAD), 0, abort_flag, p.status, kSiteConsumerFull,
                                                     p.test_stall_ns));
        auto zero_row = [&](uint32_t off) {  // this thread's 32 columns of a tile row
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4 *>(gb + off + swz(r, 4 * hh + k)) = make_uint4(0u, 0u, 0u, 0u);
        };
        // Start weights of chain bhx, thread h's rows (h = tid = TMEM lane 32q + lane of
        // weight tile hh), in four batches of 32 values: W1^T features 0-31 and 32-63,
        // then W2 features 0-31 and 32-63; they go to the weight accumulators (fp32).
        // W2 rows (this warp's 32 hidden units, 32 features a batch) pass through a
        // per-warp 2 KB piece of the Et tile, which the plain model leaves idle outside
        // the update pass, 16 features at a time: global memory then sees 64-byte row
        // pieces four lanes wide instead of one 16-byte piece per lane and row.  The
        // 16-byte chunks of a row are XOR-swizzled so both sides hit distinct banks.
        const uint32_t wstg = base + C::ET_OFF + 2048u * (uint32_t)warp;
        const int hbase = 128 * hh + 32 * q;  // this warp's first hidden unit
        auto stg_off = [](int row, int c) { return (uint32_t)row * 64u + (((uint32_t)c ^ (((uint32_t)row >> 1) & 3u)) << 4); };
        auto load_batch = [&](int bhx, int b, uint32_t (&v)[32]) {
            const size_t ps = p.per_batch ? (size_t)bhx : (size_t)(bhx % p.H);
            if (b < 2) {
                const float *w1 = p.W1 + ps * D * M + (size_t)(32 * b) * M + tid;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(w1[(size_t)j * M]);
            } else if constexpr (!LN) {  // in staging order: row 8i + lane / 4, 16-byte chunk lane % 4
                const float *w2 = p.W2 + ps * M * D + (size_t)hbase * D + 32 * (b - 2);
#pragma unroll
                for (int rho = 0; rho < 2; ++rho)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 f = *reinterpret_cast<const float4 *>(
                            w2 + (size_t)(8 * i + (lane >> 2)) * D + 16 * rho + 4 * (lane & 3));
                        v[16 * rho + 4 * i] = __float_as_uint(f.x);
                        v[16 * rho + 4 * i + 1] = __float_as_uint(f.y);
                        v[16 * rho + 4 * i + 2] = __float_as_uint(f.z);
                        v[16 * rho + 4 * i + 3] = __float_as_uint(f.w);
                    }
            } else {
                const float4 *w2 = reinterpret_cast<const float4 *>(p.W2 + ps * M * D + (size_t)tid * D) + 8 * (b - 2);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 f = w2[i];
                    v[4 * i] = __float_as_uint(f.x);
                    v[4 * i + 1] = __float_as_uint(f.y);
                    v[4 * i + 2] = __float_as_uint(f.z);
                    v[4 * i + 3] = __float_as_uint(f.w);
                }
            }
        };
        auto store_batch = [&](int b, const uint32_t (&v)[32]) {
            if (!LN && b >= 2) {  // back from staging order to this thread's row
                uint32_t rowv[32];
#pragma unroll
                for (int rho = 0; rho < 2; ++rho) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(wstg + stg_off(8 * i + (lane >> 2), lane & 3)),
                                     "r"(v[16 * rho + 4 * i]), "r"(v[16 * rho + 4 * i + 1]), "r"(v[16 * rho + 4 * i + 2]),
                                     "r"(v[16 * rho + 4 * i + 3])
                                     : "memory");
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 u = lds128(wstg + stg_off(lane, c));
                        rowv[16 * rho + 4 * c] = u.x;
                        rowv[16 * rho + 4 * c + 1] = u.y;
                        rowv[16 * rho + 4 * c + 2] = u.z;
                        rowv[16 * rho + 4 * c + 3] = u.w;
                    }
                    __syncwarp();
                }
                tc_st32(tl + C::T_W2 + 64u * hh + 32u * (uint32_t)(b & 1), rowv);
                return;
            }
            tc_st32(tl + (b < 2 ? C::T_W1 + C::W1C * hh : C::T_W2 + 64u * hh) + 32u * (uint32_t)(b & 1), v);
        };
        auto load_bias = [&](int bhx, float &c1v, float &c2v, float &lnv) {
            const size_t ps = p.per_batch ? (size_t)bhx : (size_t)(bhx % p.H);
            c1v = p.c1[ps * M + tid];
            c2v = tid < D ? p.c2[ps * D + tid] : 0.f;
            if constexpr (LN)  // thread i < 2d: gamma[i] (i < d) or beta[i - d] of the chain's head
                lnv = tid < 2 * D ? (tid < D ? p.ln_gamma : p.ln_beta)[(size_t)(bhx % p.H) * D + (tid & (D - 1))] : 0.f;
        };
        // bf16 copy of thread h's row of a weight accumulator into a [256][64] operand tile
        auto copy_row = [&](uint32_t tcol, int off) {  // tcol: the row's first column
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t wr[32];
                tc_ld32_nowait(tl + tcol + 32u * (uint32_t)half, wr);
                tc_wait_ld();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4 *>(gb + off + swz(tid, 4 * half + k)) =
                        make_uint4(pack_bf16(__uint_as_float(wr[8 * k]), __uint_as_float(wr[8 * k + 1])),
                                   pack_bf16(__uint_as_float(wr[8 * k + 2]), __uint_as_float(wr[8 * k + 3])),
                                   pack_bf16(__uint_as_float(wr[8 * k + 4]), __uint_as_float(wr[8 * k + 5])),
                                   pack_bf16(__uint_as_float(wr[8 * k + 6]), __uint_as_float(wr[8 * k + 7])));
            }
        };
        // batch b (as in load_batch) of thread h's final weights, from the accumulators to
        // W1 [d][m] (stride m: coalesced over the warp's hidden units) or W2 [m][d]
        auto store_out = [&](int bhx, int b) {
            uint32_t wr[32];
            tc_ld32_nowait(tl + (b < 2 ? C::T_W1 + C::W1C * hh : C::T_W2 + 64u * hh) + 32u * (uint32_t)(b & 1), wr);
            tc_wait_ld();
            if (b < 2) {
                if (p.W1o) {
                    float *o = p.W1o + (size_t)bhx * D * M + (size_t)(32 * b) * M + tid;
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[(size_t)j * M] = __uint_as_float(wr[j]);
                }
            } else if (p.W2o) {
                if constexpr (!LN) {  // through the staging piece, 16 features at a time
                    float *o = p.W2o + ((size_t)bhx * M + hbase) * D + 32 * (b - 2);
#pragma unroll
                    for (int rho = 0; rho < 2; ++rho) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(wstg + stg_off(lane, c)),
                                         "r"(wr[16 * rho + 4 * c]), "r"(wr[16 * rho + 4 * c + 1]),
                                         "r"(wr[16 * rho + 4 * c + 2]), "r"(wr[16 * rho + 4 * c + 3])
                                         : "memory");
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = 8 * i + (lane >> 2);
                            const uint4 u = lds128(wstg + stg_off(row, lane & 3));
                            *reinterpret_cast<uint4 *>(o + (size_t)row * D + 16 * rho + 4 * (lane & 3)) = u;
                        }
                        __syncwarp();
                    }
                } else {
                    float4 *o = reinterpret_cast<float4 *>(p.W2o + ((size_t)bhx * M + tid) * D) + 8 * (b - 2);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        o[i] = make_float4(__uint_as_float(wr[4 * i]), __uint_as_float(wr[4 * i + 1]),
                                           __uint_as_float(wr[4 * i + 2]), __uint_as_float(wr[4 * i + 3]));
                }
            }
        };
        uint32_t sp[4][16];  // act'(H) of this thread's row, 32 hidden units per chunk, packed bf16
        float c1_next = 0.f, c2_next = 0.f;  // the next chain's biases (thread h: c1[h], c2[h] for h < d)
        float ln_next = 0.f;                 // ... and inner-norm parameters (thread i < 2d)
        for (int ci = 0, bh = blockIdx.x; bh < p.BH; ++ci, bh += gridDim.x) {
            // ------------------------------------------------ start weights
            // (the first chain's are loaded here, the later ones' during the previous
            // chain's last output tile)
            named_sync_compute();  // the previous chain's reads of c1, c2 and the bf16 weights are done
            if (ok) {
                if (ci == 0) {
#pragma unroll 1
                    for (int b = 0; b < 4; ++b) {
                        uint32_t v[32];
                        load_batch(bh, b, v);
                        store_batch(b, v);
                    }
                    load_bias(bh, c1_next, c2_next, ln_next);
                    tc_st1(tl + C::T_W1 + C::W1C * hh + 64, __float_as_uint(c1_next));
                }
                tc_wait_st();
                copy_row(C::T_W1 + C::W1C * hh, C::W1_OFF);
                copy_row(C::T_W2 + 64u * hh, C::W2_OFF);
                c1s[tid] = c1_next;
                if (tid < D) c2s[tid] = c2_next;
                if (LN && tid < 2 * D) gms[tid] = ln_next;  // (bts = gms + d)
            }
            fence_proxy_async();
            named_sync_compute();  // c1, c2 visible to every warp
            release(B_WSTART);

            // ------------------------------------------------ update pass
            for (int mt = 0; mt < nt; ++mt, ++g, ++nu) {
                const int tb = R * (4 * mt + q), t = tb + lane;  // the quarter's first token; this row's
                const bool active = tb < T;                      // any token in the quarter
                const bool valid = lane < R && t < T;            // this row holds token t
                const uint32_t stg = (uint32_t)(g & 1) * C::STAGE;
#pragma unroll
                for (int c = 0; c < 4; ++c, ++jj) {  // A_c = act(H_c + c1), act'(H_c + c1)
                    wt(B_SFULL + (jj & 1), (jj >> 1) & 1, kSiteConsumerFull);
                    tc_fence_after();
                    if (ok && active) {
                        uint32_t hr[32];
                        tc_ld32_nowait(tl + C::T_SLOT + 64u * (uint32_t)(jj & 1) + 32u * (uint32_t)hh, hr);
                        tc_wait_ld();
                        const float2 *cb = reinterpret_cast<const float2 *>(c1s + 64 * c + 32 * hh);
                        uint32_t ap[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 h2 = __fadd2_rn(f2(hr[2 * i], hr[2 * i + 1]), cb[i]);
                            float2 a2, d2;
                            if constexpr (ACT == 0) {
                                silu_d2(h2, a2, d2);
                            } else {
                                gelu_vd(h2.x, a2.x, d2.x);
                                gelu_vd(h2.y, a2.y, d2.y);
                            }
                            ap[i] = pack2(a2);
                            sp[c][i] = pack2(d2);
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<uint4 *>(gb + C::A_OFF + C::TILE * c + swz(r, 4 * hh + k)) =
                                make_uint4(ap[4 * k], ap[4 * k + 1], ap[4 * k + 2], ap[4 * k + 3]);
                    } else if (ok) {
                        zero_row(C::A_OFF + C::TILE * c);
                    }
                    release(B_SFREE + (jj & 1));
                }
                // Et = -eta (E + c2 - V) on this warp's 32 columns (0 on rows without a token)
                wt(B_EFULL, ne & 1, kSiteConsumerReady);
                ++ne;
                tc_fence_after();
                if constexpr (LN) {
                    // with the inner norm the residual row is dl/dy for 1/2 ||k + LN(y) - v||^2,
                    // y = E + c2: per-token statistics over the row's 64 columns, half of them
                    // in the partner warp (exchanged through each thread's own Et chunks,
                    // which it overwrites only after a last pair barrier); the barriers run
                    // whenever the quarter holds tokens, so both partners always meet
                    if (active) {
                        const float et = valid ? (p.eta ? p.eta[(size_t)bh * T + t] : p.eta_scalar) : 0.f;
                        uint32_t er[32];
                        tc_ld32_nowait(tl + C::T_E + 32u * (uint32_t)hh, er);
                        tc_wait_ld();
                        float y[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(er[j]) + c2s[32 * hh + j];
                        auto xchg = [&](int slot, float a, float b) -> float2 {  // the partner's (a, b)
                            *reinterpret_cast<float2 *>(gb + C::ET_OFF + swz(r, 4 * hh + slot)) = make_float2(a, b);
                            named_sync_pair(q);
                            return *reinterpret_cast<const float2 *>(gb + C::ET_OFF + swz(r, 4 * (1 - hh) + slot));
                        };
                        float s1 = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) s1 += y[j];
                        const float mu = (s1 + xchg(0, s1, 0.f).x) * (1.f / D);
                        float s2 = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) s2 = fmaf(y[j] - mu, y[j] - mu, s2);
                        const float rs = rsqrtf((s2 + xchg(1, s2, 0.f).x) * (1.f / D) + p.ln_eps);
#pragma unroll
                        for (int j = 0; j < 32; ++j) y[j] = (y[j] - mu) * rs;  // yh
                        // g = gamma (k + gamma yh + beta - v), recomputed in the second sweep
                        auto g_of = [&](int j, float kj, float vj) {
                            const int jc = 32 * hh + j;
                            return gms[jc] * (kj + fmaf(gms[jc], y[j], bts[jc]) - vj);
                        };
                        float g1 = 0.f, g2 = 0.f;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint4 kk4 = *reinterpret_cast<const uint4 *>(gb + stg + swz(r, 4 * hh + k));
                            const uint4 vv4 = *reinterpret_cast<const uint4 *>(gb + stg + C::TILE + swz(r, 4 * hh + k));
                            const uint32_t kw[4] = {kk4.x, kk4.y, kk4.z, kk4.w}, vw[4] = {vv4.x, vv4.y, vv4.z, vv4.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int j = 8 * k + 2 * i;
                                const float ga = g_of(j, bf16_lo(kw[i]), bf16_lo(vw[i]));
                                const float gb2 = g_of(j + 1, bf16_hi(kw[i]), bf16_hi(vw[i]));
                                g1 += ga + gb2;
                                g2 = fmaf(ga, y[j], fmaf(gb2, y[j + 1], g2));
                            }
                        }
                        const float2 gp = xchg(2, g1, g2);
                        const float mg = (g1 + gp.x) * (1.f / D), mgy = (g2 + gp.y) * (1.f / D);
                        named_sync_pair(q);  // the partner has read this thread's exchange slots
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint4 kk4 = *reinterpret_cast<const uint4 *>(gb + stg + swz(r, 4 * hh + k));
                            const uint4 vv4 = *reinterpret_cast<const uint4 *>(gb + stg + C::TILE + swz(r, 4 * hh + k));
                            const uint32_t kw[4] = {kk4.x, kk4.y, kk4.z, kk4.w}, vw[4] = {vv4.x, vv4.y, vv4.z, vv4.w};
                            uint32_t o[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {  // -eta (g - mean g - yh mean(g yh)) / s
                                const int j = 8 * k + 2 * i;
                                const float da = (g_of(j, bf16_lo(kw[i]), bf16_lo(vw[i])) - mg - y[j] * mgy) * rs;
                                const float db = (g_of(j + 1, bf16_hi(kw[i]), bf16_hi(vw[i])) - mg - y[j + 1] * mgy) * rs;
                                o[i] = pack_bf16(-et * da, -et * db);
                            }
                            *reinterpret_cast<uint4 *>(gb + C::ET_OFF + swz(r, 4 * hh + k)) = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    } else {
                        zero_row(C::ET_OFF);
                    }
                } else if (ok && active) {
                    const float et = valid ? (p.eta ? p.eta[(size_t)bh * T + t] : p.eta_scalar) : 0.f;
                    uint32_t er[32];
                    tc_ld32_nowait(tl + C::T_E + 32u * (uint32_t)hh, er);
                    tc_wait_ld();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int ch = 4 * hh + k;
                        const uint4 vv = *reinterpret_cast<const uint4 *>(gb + stg + C::TILE + swz(r, ch));
                        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
                        uint32_t o[4];
                        const float2 *cb = reinterpret_cast<const float2 *>(c2s + 32 * hh + 8 * k);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {  // -eta (E + c2 - v)
                            const int j = 8 * k + 2 * i;
                            const float2 y = __fadd2_rn(f2(er[j], er[j + 1]), cb[i]);
                            o[i] = pack2(__fmul2_rn(__ffma2_rn(unpack2(vw[i]), make_float2(-1.f, -1.f), y),
                                                    make_float2(-et, -et)));
                        }
                        *reinterpret_cast<uint4 *>(gb + C::ET_OFF + swz(r, ch)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                } else if (ok) {
                    zero_row(C::ET_OFF);
                }
                release(B_ETREADY);
                // Dl_c = P_c .* act'(H_c), written over A_c once the W2 write has read it
#pragma unroll
                for (int c = 0; c < 4; ++c, ++jj) {
                    wt(B_SFULL + (jj & 1), (jj >> 1) & 1, kSiteConsumerFull);
                    tc_fence_after();
                    uint32_t o[16];  // (computed while the W2 write may still be reading A_c)
                    if (ok && active) {
                        uint32_t pr[32];
                        tc_ld32_nowait(tl + C::T_SLOT + 64u * (uint32_t)(jj & 1) + 32u * (uint32_t)hh, pr);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = pack2(__fmul2_rn(f2(pr[2 * i], pr[2 * i + 1]), unpack2(sp[c][i])));
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = 0u;
                    }
                    if (c == 0 || c == 2) wt(B_AFREE + c / 2, nu & 1, kSiteConsumerReady);
                    if (ok)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<uint4 *>(gb + C::A_OFF + C::TILE * c + swz(r, 4 * hh + k)) =
                                make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
                    release(B_SFREE + (jj & 1));
                }
            }

            // ------------------------------------------------ updated weights
            wt(B_WDONE, ci & 1, kSiteConsumerReady);
            tc_fence_after();
            if (ok) {  // thread h = tid owns hidden unit h (TMEM lane of weight tile hh)
                copy_row(C::T_W1 + C::W1C * hh, C::W1_OFF);  // the fp32 rows leave during the first output tile
                copy_row(C::T_W2 + 64u * hh, C::W2_OFF);
                const float c1n = tc_ld1(tl + C::T_W1 + C::W1C * hh + 64);  // seeded with c1
                c1s[tid] = c1n;
                if (p.c1o) p.c1o[(size_t)bh * M + tid] = c1n;
                if (hh == 0) {  // c2 writes: feature 16q + i in lane 32q + i, i < 16
                    const float s2 = tc_ld1(tl + C::T_C2);
                    if (lane < 16) {
                        const int j = 16 * q + lane;
                        const float c2n = c2s[j] + s2;
                        c2s[j] = c2n;
                        if (p.c2o) p.c2o[(size_t)bh * D + j] = c2n;
                    }
                }
            }
            fence_proxy_async();
            named_sync_compute();  // c1', c2' visible to every warp
            release(B_WREADY);

            // ------------------------------------------------ output pass
            for (int mt = 0; mt < nt; ++mt, ++g) {
                const int tb = R * (4 * mt + q), t = tb + lane;
                const bool active = tb < T, valid = lane < R && t < T;
                // last tile: the next chain's start weights come in batch by batch, each
                // load's latency behind one chunk, into the freed weight accumulators
                const int bhn = bh + (int)gridDim.x;
                const bool pre = mt == nt - 1 && bhn < p.BH;
                const bool wout = mt == 0;  // the final weights leave one batch per chunk
                if (pre && ok) load_bias(bhn, c1_next, c2_next, ln_next);
#pragma unroll
                for (int c = 0; c < 4; ++c, ++jj) {  // A_q,c = act(H_q,c + c1')
                    uint32_t nx[32];
                    if (pre && ok) load_batch(bhn, c, nx);
                    wt(B_SFULL + (jj & 1), (jj >> 1) & 1, kSiteConsumerFull);
                    tc_fence_after();
                    if (ok && active) {
                        uint32_t hr[32];
                        tc_ld32_nowait(tl + C::T_SLOT + 64u * (uint32_t)(jj & 1) + 32u * (uint32_t)hh, hr);
                        tc_wait_ld();
                        const float2 *cb = reinterpret_cast<const float2 *>(c1s + 64 * c + 32 * hh);
                        uint32_t ap[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 h2 = __fadd2_rn(f2(hr[2 * i], hr[2 * i + 1]), cb[i]);
                            if constexpr (ACT == 0) ap[i] = pack2(silu2(h2));
                            else ap[i] = pack_bf16(gelu_v(h2.x), gelu_v(h2.y));
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<uint4 *>(gb + C::A_OFF + C::TILE * c + swz(r, 4 * hh + k)) =
                                make_uint4(ap[4 * k], ap[4 * k + 1], ap[4 * k + 2], ap[4 * k + 3]);
                    }
                    release(B_SFREE + (jj & 1));
                    if (wout && ok) store_out(bh, c);
                    if (pre && ok) {
                        store_batch(c, nx);
                        if (c == 0) tc_st1(tl + C::T_W1 + C::W1C * hh + 64, __float_as_uint(c1_next));
                    }
                }
                // Z = the accumulated product + c2' on this warp's 32 columns
                wt(B_EFULL, ne & 1, kSiteConsumerReady);
                ++ne;
                tc_fence_after();
                if constexpr (LN) {  // z = q + LN(y), y = Z + c2' (the idle Et tile carries the exchange)
                    if (active) {
                        uint32_t zr[32];
                        tc_ld32_nowait(tl + C::T_E + 32u * (uint32_t)hh, zr);
                        tc_wait_ld();
                        float y[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(zr[j]) + c2s[32 * hh + j];
                        auto xchg = [&](int slot, float a) -> float {
                            *reinterpret_cast<float *>(gb + C::ET_OFF + swz(r, 4 * hh + slot)) = a;
                            named_sync_pair(q);
                            return *reinterpret_cast<const float *>(gb + C::ET_OFF + swz(r, 4 * (1 - hh) + slot));
                        };
                        float s1 = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) s1 += y[j];
                        const float mu = (s1 + xchg(0, s1)) * (1.f / D);
                        float s2 = 0.f;
#pragma unroll
                        for (int j = 0; j < 32; ++j) s2 = fmaf(y[j] - mu, y[j] - mu, s2);
                        const float rs = rsqrtf((s2 + xchg(1, s2)) * (1.f / D) + p.ln_eps);
                        if (valid && ok) {
                            const uint4 *qr = reinterpret_cast<const uint4 *>(p.q + ((size_t)bh * T + t) * D + 32 * hh);
                            uint4 *dst = reinterpret_cast<uint4 *>(p.z + ((size_t)bh * T + t) * D + 32 * hh);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint4 q4 = qr[k];
                                const uint32_t qw[4] = {q4.x, q4.y, q4.z, q4.w};
                                uint32_t o[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int j = 8 * k + 2 * i, jc = 32 * hh + j;
                                    o[i] = pack_bf16(bf16_lo(qw[i]) + fmaf(gms[jc], (y[j] - mu) * rs, bts[jc]),
                                                     bf16_hi(qw[i]) + fmaf(gms[jc + 1], (y[j + 1] - mu) * rs, bts[jc + 1]));
                                }
                                dst[k] = make_uint4(o[0], o[1], o[2], o[3]);
                            }
                        }
                        named_sync_pair(q);  // the exchange slots are free again
                    }
                } else if (ok && active) {
                    uint32_t zr[32];
                    tc_ld32_nowait(tl + C::T_E + 32u * (uint32_t)hh, zr);
                    tc_wait_ld();
                    if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.z + ((size_t)bh * T + t) * D + 32 * hh);
                        const float2 *cb = reinterpret_cast<const float2 *>(c2s + 32 * hh);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int j = 8 * k;
                            dst[k] = make_uint4(pack2(__fadd2_rn(f2(zr[j], zr[j + 1]), cb[j / 2])),
                                                pack2(__fadd2_rn(f2(zr[j + 2], zr[j + 3]), cb[j / 2 + 1])),
                                                pack2(__fadd2_rn(f2(zr[j + 4], zr[j + 5]), cb[j / 2 + 2])),
                                                pack2(__fadd2_rn(f2(zr[j + 6], zr[j + 7]), cb[j / 2 + 3])));
                        }
                    }
                }
                tc_fence_before();
            }
        }
        tc_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::NCW) tc_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace

// One non-causal full-batch mini-batch (b >= T >= 1), d = 64, m = 256, bf16, with or
// without the inner norm; -2 otherwise.
int launch_mlp_fb_tc(const MlpArgs &a)
{
    using C = FmtCfg;
    if (a.d != 64 || a.m != 256 || a.causal || a.b < a.T || a.T < 1) return -2;
    CUtensorMap maps[3];
    if (!encode_qkv(maps, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 32)) return -4;  // 32-row boxes
    auto kern = a.ln_gamma ? (a.act ? ttt_mlp_fb_tc_kernel<1, true> : ttt_mlp_fb_tc_kernel<0, true>)
                           : (a.act ? ttt_mlp_fb_tc_kernel<1, false> : ttt_mlp_fb_tc_kernel<0, false>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return -4;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -4;
    FmtParams p;
    p.BH = a.B * a.H;
    p.H = a.H;
    p.T = a.T;
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
    p.test_stall_ns = a.test_stall_ns;
    const int grid = p.BH < nsm ? p.BH : nsm;
    kern<<<grid, C::THREADS, C::SMEM, a.stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace ttt
