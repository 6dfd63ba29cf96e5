// ttt_linear_blk.cu -- causal TTT-Linear with mini-batches of 16 tokens, d = 64, bf16
// operands, fp32 state: the block form on the 5th-generation tensor cores.
//
// The layer ("Learning to (Learn at Test Time)" walkthrough, section 1.2.2, mini-batch
// gradient descent and its dual form; "Fast weights 与 TTT layers", section 2, updates
// taken in blocks for hardware utilisation).  Take a block of 64 tokens = four
// mini-batches i = 0..3 with start weights W.  The step of token s in mini-batch i is
// u_s = -eta_s (k_s W_i - v_s), W_i = W + sum_{j<i} K_j^T U_j, so the steps U of the
// block solve the block-unit-lower-triangular system
//     (I + L) U = diag(eta) (V - K W),   L_ij = diag(eta_i) K_i K_j^T  (j < i, else 0)
// and with Tt = (I + L)^-1 diag(eta), P = -Tt K, C = Tt V:  U = P W + C.  Then
//     W_next = W + X W + B,      X = K^T P,  B = K^T C
//     Z      = Q' W + C',        Q' = Q + tril(Q K^T) P,  C' = tril(Q K^T) C
// (tril keeps key s <= query t over the whole block: z_t reads the writes of the
// earlier mini-batches of the block and of its own tokens up to t).  Only the product
// [Q'; X] W of each block depends on the state; everything else is formed from the
// block's inputs, ahead of time.  L is nilpotent (L^4 = 0), so (I + L)^-1 is exact by
// block forward substitution over the 16 x 16 blocks.
//
// One CTA per (batch, head) chain, one per SM (210 KB of shared memory, 512 columns
// of tensor memory), eleven warps:
//  * warp 8 streams each block's K, Q, V by TMA (64-token boxes, 128-byte swizzle) into
//    a ring of five slots, and its rates eta by 4-byte copies;
//  * warp 9 (one thread) issues the tcgen05 products, each a 128-row M from shared
//    memory into tensor memory, and commits each to an mbarrier:
//        P1 = [K; Q] K^T                 (G = K K^T and S = Q K^T)
//        Mt = -[tril(S); K^T] Tt         (M = 128, K over the block's tokens)
//        F  = Mt [K | V]                 (two N = 64 products: [Q' - Q | -C'; X | -B])
//        CH = [Q'; X] W_bf16             (the chain: rows 0-63 Q'W, rows 64-127 XW)
//  * warp 10 forms -Tt^T from L with mma.sync (eight 16 x 16 x 16 products) and writes
//    it as the K-major B operand of Mt;
//  * warps 0-7 own tensor-memory lanes 32 (w % 4) .. +31 and columns 32 (w / 4) .. +31 of
//    each 64-column result; they run the epilogues: masks and eta scaling of P1 (L and
//    tril(S)), K^T by ldmatrix.trans / stmatrix, the bf16 copies of Mt and F, Q' = Q +
//    (Q' - Q), and the chain epilogue: z = Q'W + C' to global memory and W += XW + B in
//    fp32 registers (threads of lanes 64-127 hold W's rows), whose bf16 copy is the next
//    chain product's B operand.
// The epilogue warps run, per step n, E_Mt(n+2), E_P1(n+3), E_CH(n) and E_F(n+1): every
// product they wait for was issued a stage or more before, so the tensor core works on
// later blocks while they run, and the serial chain costs one product per 64 tokens.
//
// Every wait is bounded (kWaitLimitNs); the first to run out records its site in the
// status word and raises a shared abort flag that ends every other wait, after which
// the producer waits for its copies in flight, the issuing thread for its products, and
// warp 0 frees the tensor memory.
#include <cuda.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"
#include "ttt_tcgen05.cuh"

namespace ttt {
namespace {

struct BlkCfg {
    static constexpr int D = 64;
    static constexpr int NEPI = 16;                      // epilogue warps
    static constexpr int CW = 64 / (NEPI / 4);           // columns per epilogue warp
    static constexpr int NCH = CW / 8;                   // 16-byte bf16 chunks per row slice
    static constexpr int WP = 16, WM = 17, WT = 18, WC = 19;  // producer, issuers, inverse warp
    static constexpr int THREADS = 20 * 32;
    static constexpr int NS = 5;                         // input slots: K | Q | V of a block
    static constexpr int ND = 3;                         // derived buffers [tril(S); K^T] -> Mt
    static constexpr int TILE = 64 * 128;                // 64 rows of 64 bf16
    static constexpr int SLOT = 3 * TILE;
    static constexpr int DER_OFF = NS * SLOT;
    static constexpr int CH_OFF = DER_OFF + ND * 2 * TILE;  // [Q'; X], the chain's A operand
    static constexpr int L_OFF = CH_OFF + 2 * TILE;         // L (rows t, columns s), bf16
    static constexpr int T_OFF = L_OFF + TILE;              // -Tt^T (rows u, columns s), bf16, two buffers
    static constexpr int W_OFF = T_OFF + 2 * TILE;          // W (rows i), bf16: the chain's B
    static constexpr int ETA_OFF = W_OFF + TILE;            // NS x 64 fp32
    static constexpr int BAR_OFF = ETA_OFF + NS * 256;
    // B_A: one per derived buffer, B_T and B_MT one per -Tt^T buffer (their waiters may be
    // a block apart, so a single barrier could complete twice before one of them looks)
    enum { B_FULL = 0, B_EMPTY = NS, B_A = 2 * NS, B_T = B_A + ND, B_MT = B_T + 2, B_P1 = B_MT + 2, B_B, B_L, B_CH,
           B_F, B_C, B_FIN, B_FIN2, NBAR };
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;     // tensor-memory address, abort flag
    static constexpr int SMEM = MISC_OFF + 16 + 1024;       // + slack for the 1024-byte alignment
    static constexpr int TMEM_COLS = 512;
    // tensor-memory columns: F is double-buffered (block j at C_F + 128 (j % 2)): its V
    // half is read by the chain epilogue of block j while F(j+1) is already formed
    static constexpr uint32_t C_P1 = 0, C_MT = 64, C_F = 128, C_CH = 384;
};
static_assert(BlkCfg::SMEM <= 227 * 1024, "shared memory");

struct BlkParams {
    int H, T;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    __nv_bfloat16 *z;
    float *W_out;
    int *status;
};

// Byte offset of 16-byte chunk ch of row r in a tile of 128-byte rows with the
// 128-byte swizzle (the layout TMA writes and the tensor core reads).
__device__ __forceinline__ uint32_t swz(int r, int ch) { return (uint32_t)(r * 128 + ((ch ^ (r & 7)) << 4)); }

__device__ __forceinline__ void st128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Bounded wait that also ends when another role has given up (shared abort flag).
__device__ __forceinline__ bool blk_wait(uint32_t bar, uint32_t parity, int *status, volatile int *abort_flag,
                                         int site)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                atomicCAS(status, 0, site);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__global__ void __launch_bounds__(BlkCfg::THREADS, 1)
    ttt_linear_blk_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                             const __grid_constant__ CUtensorMap tv, const BlkParams p)
{
    using C = BlkCfg;
    constexpr int D = C::D, NS = C::NS, ND = C::ND;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gb = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, T = p.T;
    const int nblk = (T + 63) >> 6;
    const bool has_eta = p.eta != nullptr;
    const uint32_t bar0 = base + C::BAR_OFF;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gb + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(gb + C::MISC_OFF + 8);
    const float *etas = reinterpret_cast<const float *>(gb + C::ETA_OFF);
    auto slot_of = [&](int j) { return base + (uint32_t)((j % NS) * C::SLOT); };  // K at +0, Q +TILE, V +2 TILE
    auto der_of = [&](int j) { return base + C::DER_OFF + (uint32_t)((j % ND) * 2 * C::TILE); };
    const uint32_t sCH = base + C::CH_OFF, sL = base + C::L_OFF, sT = base + C::T_OFF, sW = base + C::W_OFF;
    // the rate of token u of block j (zero past the sequence, so padded rows stay inert)
    auto eta_at = [&](int j, int u) -> float {
        const int tok = 64 * j + u;
        return tok < T ? (has_eta ? etas[(j % NS) * 64 + u] : p.eta_scalar) : 0.f;
    };

    if (tid == 0) {
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(C::B_FULL + s), 1 + (has_eta ? 32 : 0));
            mbar_init(bar(C::B_EMPTY + s), C::NEPI);
        }
        mbar_init(bar(C::B_P1), 1);
        for (int r = 0; r < 2; ++r) {
            mbar_init(bar(C::B_MT + r), 1);
            mbar_init(bar(C::B_T + r), 1);
        }
        for (int r = 0; r < ND; ++r) mbar_init(bar(C::B_A + r), C::NEPI);
        mbar_init(bar(C::B_B), C::NEPI);
        mbar_init(bar(C::B_L), C::NEPI);
        mbar_init(bar(C::B_CH), 1);
        mbar_init(bar(C::B_F), 1);
        mbar_init(bar(C::B_C), C::NEPI);
        mbar_init(bar(C::B_FIN), 1);
        mbar_init(bar(C::B_FIN2), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tc_alloc(base + C::MISC_OFF, C::TMEM_COLS);
    // -Tt^T: the blocks above the block diagonal stay zero for the whole run
    for (int i = tid; i < 2 * C::TILE / 16; i += C::THREADS) st128(sT + 16 * i, 0, 0, 0, 0);

    // epilogue warps: quarter qw of the tensor-memory lanes, columns cb .. cb + CW - 1
    constexpr int CW = C::CW, NCH = C::NCH;
    const int qw = warp & 3, cb = CW * (warp >> 2), chb = cb / 8, r = 32 * qw + lane;
    const bool wrow = warp < C::NEPI && r >= 64;  // holds row i = r - 64 of W (fp32)
    const int wi = r - 64;
    float Wr[CW];
    if (wrow) {
        const float *W0 = p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * D * D +
                          (size_t)wi * D + cb;
#pragma unroll
        for (int e = 0; e < CW; ++e) Wr[e] = W0[e];
#pragma unroll
        for (int c = 0; c < NCH; ++c)
            st128(sW + swz(wi, chb + c), pack_bf16(Wr[8 * c], Wr[8 * c + 1]), pack_bf16(Wr[8 * c + 2], Wr[8 * c + 3]),
                  pack_bf16(Wr[8 * c + 4], Wr[8 * c + 5]), pack_bf16(Wr[8 * c + 6], Wr[8 * c + 7]));
    }
    fence_proxy_async();  // W_bf16 and the zero blocks of -Tt^T before the tensor core reads them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool ok = true;

    if (warp == C::WP) {
        // ---------------------------------------------------------------- producer
        int issued = 0;
        for (int j = 0; j < nblk && ok; ++j) {
            const int s = j % NS;
            if (j >= NS) ok = blk_wait(bar(C::B_EMPTY + s), ((j / NS) & 1) ^ 1, p.status, abort_flag, kSiteProducerEmpty);
            if (!ok) break;
            const uint32_t full = bar(C::B_FULL + s), st = slot_of(j);
            if (has_eta) {
                const uint32_t ed = base + C::ETA_OFF + s * 256;
#pragma unroll
                for (int i = lane; i < 64; i += 32)
                    if (64 * j + i < T) cp_async_4(ed + 4 * i, p.eta + (size_t)bh * T + 64 * j + i);
                cp_async_arrive_noinc(full);
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(full, 3 * C::TILE);
                tma_load_3d(st, &tk, full, 0, 64 * j, bh);
                tma_load_3d(st + C::TILE, &tq, full, 0, 64 * j, bh);
                tma_load_3d(st + 2 * C::TILE, &tv, full, 0, 64 * j, bh);
            }
            __syncwarp();
            issued = j + 1;
        }
        // copies still in flight end before the CTA does
        for (int j = issued > NS ? issued - NS : 0; j < issued; ++j)
            if (!mbar_wait(bar(C::B_FULL + j % NS), (j / NS) & 1, p.status, kSiteDrain)) break;
    } else if (warp == C::WM) {
        // ------------------------------------------- issuer of the input-only products
        if (lane == 0) {
            constexpr uint32_t idKK = idesc_bf16(128, 64, false, false);
            // after part 1 of epilogue step m (E_Mt(m+1), E_P1(m+3)): P1(m+4) as soon as P1's
            // tensor memory is free, then Mt(m+2) once its -Tt^T is ready (formed a step before)
            for (int m = -4; m < nblk && ok; ++m) {
                const int jP = m + 4, jM = m + 2;
                if (jP >= 0 && jP < nblk) {  // P1 = [K; Q] K^T
                    if (jP >= 1) ok = blk_wait(bar(C::B_B), (jP - 1) & 1, p.status, abort_flag, kSiteStage);
                    ok = ok && blk_wait(bar(C::B_FULL + jP % NS), (jP / NS) & 1, p.status, abort_flag, kSiteConsumerFull);
                    if (ok) {
                        tc_fence_after();
                        const uint32_t sk = slot_of(jP);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(tmem + C::C_P1, sdesc(sk + 32 * kk, 16), sdesc(sk + 32 * kk, 16), idKK, kk > 0);
                        tc_commit(bar(C::B_P1));
                    }
                }
                if (ok && jM >= 0 && jM < nblk) {  // Mt = -[tril(S); K^T] Tt
                    if (jM >= 1)  // Mt's tensor memory has been read (E_Mt(jM-1))
                        ok = blk_wait(bar(C::B_A + (jM - 1) % ND), ((jM - 1) / ND) & 1, p.status, abort_flag, kSiteStage);
                    ok = ok && blk_wait(bar(C::B_T + (jM & 1)), (jM >> 1) & 1, p.status, abort_flag, kSiteStage);
                    if (ok) {
                        tc_fence_after();
                        const uint32_t a = der_of(jM), t = sT + (uint32_t)((jM & 1) * C::TILE);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(tmem + C::C_MT, sdesc(a + 32 * kk, 16), sdesc(t + 32 * kk, 16), idKK, kk > 0);
                        tc_commit(bar(C::B_MT + (jM & 1)));
                    }
                }
            }
            // every product issued has completed before the tensor memory is freed
            tc_commit(bar(C::B_FIN));
            mbar_wait(bar(C::B_FIN), 0, p.status, kSiteDrain);
        }
    } else if (warp == C::WC) {
        // ------------------------------------------- issuer of the chain and of F
        if (lane == 0) {
            constexpr uint32_t idKM = idesc_bf16(128, 64, false, true);
            constexpr uint32_t idF = idesc_bf16(128, 128, false, true);
            // F(j) once Mt(j) is in bf16 (part 1 of step j-1); the chain product j once Q', X
            // and W_bf16 of block j are written (part 2 of step j-1)
            for (int j = 0; j < nblk && ok; ++j) {
                ok = blk_wait(bar(C::B_A + j % ND), (j / ND) & 1, p.status, abort_flag, kSiteStage) &&
                     blk_wait(bar(C::B_FULL + j % NS), (j / NS) & 1, p.status, abort_flag, kSiteConsumerFull);
                if (!ok) break;
                {  // F = Mt [K | V]: N = 128, the K and V tiles 2 TILE apart
                    tc_fence_after();
                    const uint32_t a = der_of(j), sk = slot_of(j);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma(tmem + C::C_F + 128 * (j & 1), sdesc(a + 32 * kk, 16), sdesc(sk + 2048 * kk, 2 * C::TILE),
                               idF, kk > 0);
                    tc_commit(bar(C::B_F));
                }
                ok = blk_wait(bar(C::B_C), j & 1, p.status, abort_flag, kSiteStage);
                if (!ok) break;
                {  // the chain: [Q'; X] W
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma(tmem + C::C_CH, sdesc(sCH + 32 * kk, 16), sdesc(sW + 2048 * kk, 8192), idKM, kk > 0);
                    tc_commit(bar(C::B_CH));
                }
            }
            tc_commit(bar(C::B_FIN2));
            mbar_wait(bar(C::B_FIN2), 0, p.status, kSiteDrain);
        }
    } else if (warp == C::WT) {
        // ------------------------------------- -Tt^T from L (block forward substitution)
        const int g = lane >> 2, t4 = lane & 3;
        // ldmatrix row addresses of the 16 x 16 block at (16 bi, 16 bj): B pattern (rows
        // 0-7 / 8-15 by lane >> 4, column halves by bit 3) and A pattern for the stores
        auto addrB = [&](uint32_t tile, int bi, int bj) {
            const int row = 16 * bi + (lane & 7) + 8 * (lane >> 4);
            return tile + swz(row, 2 * bj + ((lane >> 3) & 1));
        };
        auto addrA = [&](uint32_t tile, int bi, int bj) {
            const int row = 16 * bi + (lane & 7) + 8 * ((lane >> 3) & 1);
            return tile + swz(row, 2 * bj + (lane >> 4));
        };
        for (int j = 0; j < nblk && ok; ++j) {
            ok = blk_wait(bar(C::B_L), j & 1, p.status, abort_flag, kSiteStage) &&
                 blk_wait(bar(C::B_FULL + j % NS), (j / NS) & 1, p.status, abort_flag, kSiteConsumerFull);
            // buffer j % 2 is free once Mt(j-2) has read it
            if (ok && j >= 2) ok = blk_wait(bar(C::B_MT + (j & 1)), ((j - 2) >> 1) & 1, p.status, abort_flag, kSiteStage);
            if (!ok) break;
            float er[4][2];  // -eta of rows g and g + 8 of each 16-token block
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                er[J][0] = -eta_at(j, 16 * J + g);
                er[J][1] = -eta_at(j, 16 * J + g + 8);
            }
            // L_ab^T as A fragments (ldmatrix.trans of block (a, b)); their negation is the
            // first term of A_ab = (T_ab)^T
            uint32_t l10[4], l20[4], l21[4], l30[4], l31[4], l32[4], b21[4], b31[4], b32[4];
            ldsm_x4_t(addrB(sL, 1, 0), l10[0], l10[1], l10[2], l10[3]);
            ldsm_x4_t(addrB(sL, 2, 0), l20[0], l20[1], l20[2], l20[3]);
            ldsm_x4_t(addrB(sL, 2, 1), l21[0], l21[1], l21[2], l21[3]);
            ldsm_x4_t(addrB(sL, 3, 0), l30[0], l30[1], l30[2], l30[3]);
            ldsm_x4_t(addrB(sL, 3, 1), l31[0], l31[1], l31[2], l31[3]);
            ldsm_x4_t(addrB(sL, 3, 2), l32[0], l32[1], l32[2], l32[3]);
            // L_ik^T as B fragments (ldmatrix of block (i, k)): n-tile 0 in [0..1], 1 in [2..3]
            ldsm_x4(addrB(sL, 2, 1), b21[0], b21[1], b21[2], b21[3]);
            ldsm_x4(addrB(sL, 3, 1), b31[0], b31[1], b31[2], b31[3]);
            ldsm_x4(addrB(sL, 3, 2), b32[0], b32[1], b32[2], b32[3]);
            // accumulators (two n-tiles of 16 x 8) initialised to -L_ab^T
            auto negc = [&](const uint32_t (&a)[4], float (&c)[2][4]) {
                c[0][0] = -bf16_lo(a[0]); c[0][1] = -bf16_hi(a[0]); c[0][2] = -bf16_lo(a[1]); c[0][3] = -bf16_hi(a[1]);
                c[1][0] = -bf16_lo(a[2]); c[1][1] = -bf16_hi(a[2]); c[1][2] = -bf16_lo(a[3]); c[1][3] = -bf16_hi(a[3]);
            };
            float A10[2][4], A21[2][4], A32[2][4], A20[2][4], A31[2][4], A30[2][4];
            negc(l10, A10);
            negc(l21, A21);
            negc(l32, A32);
            negc(l20, A20);
            negc(l31, A31);
            negc(l30, A30);
            // A_ij = -L_ij^T - sum_{j<k<i} A_kj L_ik^T; -A_10 = L_10^T and -A_21 = L_21^T are
            // the loaded fragments themselves
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                mma_bf16(A20[nt], l10[0], l10[1], l10[2], l10[3], b21[2 * nt], b21[2 * nt + 1]);
                mma_bf16(A31[nt], l21[0], l21[1], l21[2], l21[3], b32[2 * nt], b32[2 * nt + 1]);
                mma_bf16(A30[nt], l10[0], l10[1], l10[2], l10[3], b31[2 * nt], b31[2 * nt + 1]);
            }
            const uint32_t n20[4] = {pack_bf16(-A20[0][0], -A20[0][1]), pack_bf16(-A20[0][2], -A20[0][3]),
                                     pack_bf16(-A20[1][0], -A20[1][1]), pack_bf16(-A20[1][2], -A20[1][3])};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_bf16(A30[nt], n20[0], n20[1], n20[2], n20[3], b32[2 * nt], b32[2 * nt + 1]);
            // block (row J, column I) of -Tt^T is -diag(eta_J) A_IJ (I > J), -diag(eta_J) on
            // the diagonal
            const uint32_t sTj = sT + (uint32_t)((j & 1) * C::TILE);
            auto store = [&](const float (&c)[2][4], int J, int I) {
                const float e0 = er[J][0], e1 = er[J][1];
                stsm_x4(addrA(sTj, J, I), pack_bf16(e0 * c[0][0], e0 * c[0][1]), pack_bf16(e1 * c[0][2], e1 * c[0][3]),
                        pack_bf16(e0 * c[1][0], e0 * c[1][1]), pack_bf16(e1 * c[1][2], e1 * c[1][3]));
            };
            store(A10, 0, 1);
            store(A21, 1, 2);
            store(A32, 2, 3);
            store(A20, 0, 2);
            store(A31, 1, 3);
            store(A30, 0, 3);
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                // the identity block in accumulator layout: (g, 2 t4 + e) of n-tile 0 and
                // (g + 8, 8 + 2 t4 + e) of n-tile 1 lie on the diagonal when g = 2 t4 + e
                const float d0 = (g == 2 * t4) ? 1.f : 0.f, d1 = (g == 2 * t4 + 1) ? 1.f : 0.f;
                const float dg[2][4] = {{d0, d1, 0.f, 0.f}, {0.f, 0.f, d0, d1}};
                store(dg, J, J);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_T + (j & 1)));
        }
    } else {
        // --------------------------------------------------------- epilogue warps
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qw) << 16) + cb;
        auto f = [](uint32_t u) { return __uint_as_float(u); };
        for (int n = -3; n < nblk && ok; ++n) {
            // ---- part 1, off the chain: Mt(n+1) -> bf16 Mt (F's A operand); P1(n+3) -> L,
            //      tril(S), K^T (one proxy fence for both).  L is written once -Tt^T(n+2) has
            //      been formed from the previous one.
            const int jA = n + 1, jB = n + 3;
            const bool va = jA >= 0 && jA < nblk, vb = jB >= 0 && jB < nblk;
            if (va) ok = blk_wait(bar(C::B_MT + (jA & 1)), (jA >> 1) & 1, p.status, abort_flag, kSiteConsumerReady);
            if (ok && vb)
                ok = blk_wait(bar(C::B_P1), jB & 1, p.status, abort_flag, kSiteConsumerReady) &&
                     blk_wait(bar(C::B_FULL + jB % NS), (jB / NS) & 1, p.status, abort_flag, kSiteConsumerFull);
            if (ok && vb && jB >= 1)
                ok = blk_wait(bar(C::B_T + ((jB - 1) & 1)), ((jB - 1) >> 1) & 1, p.status, abort_flag, kSiteStage);
            if (!ok) break;
            if (va || vb) {
                tc_fence_after();
                if (va) {
                    uint32_t vu[CW];
                    tc_ld16_nowait(lane_base + C::C_MT, vu);
                    tc_wait_ld();
                    float v[CW];
#pragma unroll
                    for (int e = 0; e < CW; ++e) v[e] = f(vu[e]);
                    const uint32_t dst = der_of(jA);
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        st128(dst + swz(r, chb + c), pack_bf16(v[8 * c], v[8 * c + 1]), pack_bf16(v[8 * c + 2], v[8 * c + 3]),
                              pack_bf16(v[8 * c + 4], v[8 * c + 5]), pack_bf16(v[8 * c + 6], v[8 * c + 7]));
                }
                if (vb) {
                    uint32_t gu[CW];
                    tc_ld16_nowait(lane_base + C::C_P1, gu);
                    tc_wait_ld();
                    float g[CW];
#pragma unroll
                    for (int e = 0; e < CW; ++e) g[e] = f(gu[e]);
                    const uint32_t dst = der_of(jB);
                    if (r < 64) {  // row t of G = K K^T: L[t][s] = eta_t G[t][s] below the block diagonal
                        const int t = r, mb = t >> 4;
                        const float et = eta_at(jB, t);
#pragma unroll
                        for (int c = 0; c < NCH; ++c)
                            if (chb + c < 2 * mb)
                                st128(sL + swz(t, chb + c), pack_bf16(et * g[8 * c], et * g[8 * c + 1]),
                                      pack_bf16(et * g[8 * c + 2], et * g[8 * c + 3]),
                                      pack_bf16(et * g[8 * c + 4], et * g[8 * c + 5]),
                                      pack_bf16(et * g[8 * c + 6], et * g[8 * c + 7]));
                    } else {  // row t of S = Q K^T: tril(S)[t][s] = S[t][s] for s <= t
                        const int t = r - 64;
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            const int s0 = cb + 8 * c;
                            float m[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) m[e] = (s0 + e <= t) ? g[8 * c + e] : 0.f;
                            st128(dst + swz(t, chb + c), pack_bf16(m[0], m[1]), pack_bf16(m[2], m[3]),
                                  pack_bf16(m[4], m[5]), pack_bf16(m[6], m[7]));
                        }
                    }
                    // K^T (rows 64-127 of the derived buffer) by transposed 8 x 8 copies: warp w
                    // takes rows 8 (w % 8) .. +7 and the four token blocks 4 (w / 8) .. +3
                    const uint32_t sk = slot_of(jB);
                    const int bi = warp & 7, bt = 4 * (warp >> 3) + (lane >> 3);
                    uint32_t x0, x1, x2, x3;
                    ldsm_x4_t(sk + swz(8 * bt + (lane & 7), bi), x0, x1, x2, x3);
                    stsm_x4(dst + swz(64 + 8 * bi + (lane & 7), bt), x0, x1, x2, x3);
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (vb) {
                        mbar_arrive(bar(C::B_L));
                        mbar_arrive(bar(C::B_B));
                    }
                    if (va) mbar_arrive(bar(C::B_A + jA % ND));
                }
            }
            // ---- part 2, the chain: CH(n) and F(n)'s V half -> z = Q'W + C', W += XW + B;
            //      F(n+1)'s K half -> Q' and X, the next chain product's A operand
            const int jE = n + 1;
            const bool vd = n >= 0, vc = jE >= 0 && jE < nblk;
            if (vd) ok = blk_wait(bar(C::B_CH), n & 1, p.status, abort_flag, kSiteConsumerReady);
            if (ok && vc)
                ok = blk_wait(bar(C::B_F), jE & 1, p.status, abort_flag, kSiteConsumerReady) &&
                     blk_wait(bar(C::B_FULL + jE % NS), (jE / NS) & 1, p.status, abort_flag, kSiteConsumerFull);
            if (!ok) break;
            if (vd || vc) {
                tc_fence_after();
                if (vd) {
                    uint32_t xu[CW], uu[CW];
                    tc_ld16_nowait(lane_base + C::C_CH, xu);
                    tc_ld16_nowait(lane_base + C::C_F + 128 * (n & 1) + 64, uu);  // -C' or -B of block n
                    tc_wait_ld();
                    float x[CW];
#pragma unroll
                    for (int e = 0; e < CW; ++e) x[e] = f(xu[e]) - f(uu[e]);  // Q'W + C' (rows t) or XW + B (rows i)
                    if (r < 64) {
                        const int tok = 64 * n + r;
                        if (tok < T) {
                            uint4 *zr = reinterpret_cast<uint4 *>(p.z + ((size_t)bh * T + tok) * D + cb);
#pragma unroll
                            for (int c = 0; c < NCH; ++c)
                                zr[c] = make_uint4(pack_bf16(x[8 * c], x[8 * c + 1]), pack_bf16(x[8 * c + 2], x[8 * c + 3]),
                                                   pack_bf16(x[8 * c + 4], x[8 * c + 5]), pack_bf16(x[8 * c + 6], x[8 * c + 7]));
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < CW; ++e) Wr[e] += x[e];
#pragma unroll
                        for (int c = 0; c < NCH; ++c)
                            st128(sW + swz(wi, chb + c), pack_bf16(Wr[8 * c], Wr[8 * c + 1]),
                                  pack_bf16(Wr[8 * c + 2], Wr[8 * c + 3]), pack_bf16(Wr[8 * c + 4], Wr[8 * c + 5]),
                                  pack_bf16(Wr[8 * c + 6], Wr[8 * c + 7]));
                    }
                }
                if (vc) {
                    uint32_t yu[CW];
                    tc_ld16_nowait(lane_base + C::C_F + 128 * (jE & 1), yu);
                    tc_wait_ld();
                    float y[CW];
#pragma unroll
                    for (int e = 0; e < CW; ++e) y[e] = f(yu[e]);
                    if (r < 64) {
                        const uint32_t sq = slot_of(jE) + C::TILE;
                        uint4 qq[NCH];
#pragma unroll
                        for (int c = 0; c < NCH; ++c) qq[c] = lds128(sq + swz(r, chb + c));
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            const uint32_t qw4[4] = {qq[c].x, qq[c].y, qq[c].z, qq[c].w};
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                o[e] = pack_bf16(bf16_lo(qw4[e]) + y[8 * c + 2 * e], bf16_hi(qw4[e]) + y[8 * c + 2 * e + 1]);
                            st128(sCH + swz(r, chb + c), o[0], o[1], o[2], o[3]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < NCH; ++c)
                            st128(sCH + swz(r, chb + c), pack_bf16(y[8 * c], y[8 * c + 1]), pack_bf16(y[8 * c + 2], y[8 * c + 3]),
                                  pack_bf16(y[8 * c + 4], y[8 * c + 5]), pack_bf16(y[8 * c + 6], y[8 * c + 7]));
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && vc) {
                    mbar_arrive(bar(C::B_C));
                    mbar_arrive(bar(C::B_EMPTY + jE % NS));
                }
            }
        }
        if (ok && wrow && p.W_out) {
            float *Wo = p.W_out + (size_t)bh * D * D + (size_t)wi * D + cb;
#pragma unroll
            for (int e = 0; e < CW; ++e) Wo[e] = Wr[e];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tc_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace

// Causal, mini-batch 16, d = 64, bf16, MSE loss, one epoch, no inner norm; -2 otherwise.
int launch_linear_blk_tc(const LinearArgs &a)
{
    using C = BlkCfg;
    if (a.d != 64 || !a.causal || a.b != 16 || a.loss != 0 || a.epochs != 1 || a.ln_gamma) return -2;
    CUtensorMap maps[3];
    if (!encode_qkv(maps, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 64)) return -4;
    if (cudaFuncSetAttribute(ttt_linear_blk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
        return -4;
    BlkParams p;
    p.H = a.H;
    p.T = a.T;
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W0 = a.W0;
    p.w0_bstride = a.w0_bstride;
    p.z = static_cast<__nv_bfloat16 *>(a.z);
    p.W_out = a.W_out;
    p.status = a.status;
    ttt_linear_blk_tc_kernel<<<a.B * a.H, C::THREADS, C::SMEM, a.stream>>>(maps[0], maps[1], maps[2], p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace ttt
