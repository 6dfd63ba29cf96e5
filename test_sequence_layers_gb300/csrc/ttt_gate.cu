// ttt_gate.cu -- the input-dependent inner learning rate of a TTT layer:
//     eta[b,h,t] = eta_base * sigma(theta[h] . x[b,t])
// ("Learning to (Learn at Test Time)" walkthrough, section 2.2.3: the rate becomes a
// function of the input token through a learnable vector and a sigmoid, scaled by a
// base rate), for every head at once.  It is a product of the tokens [B*T, dm] with
// the heads' vectors [H, dm]^T, bound by reading x once from HBM (2 dm bytes per
// token against 4 H bytes of output), on mma.sync:
//  * one CTA per 64 tokens of one sequence; a producer warp streams 64-feature slices
//    of x (64 x 64 bf16) and of theta (HP x 64 bf16, rows past H zero-filled) by TMA
//    with the 128-byte swizzle through a ring of NS stages;
//  * four warps of 16 tokens each multiply their A fragments of x with B fragments of
//    theta into HP / 8 fp32 accumulator tiles, then apply eta_base * sigma and store
//    eta in the [B, H, T] layout the TTT-Linear and TTT-MLP kernels read.
#include <cuda.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

template <int HP>
struct GateCfg {
    static constexpr int THREADS = 5 * 32, PW = 4;  // four compute warps, one producer
    static constexpr int NS = 4;                      // stages in flight
    static constexpr int XB = 64 * 128;               // x slice: 64 tokens x 128 bytes
    static constexpr int STAGE = ((XB + HP * 128 + 1023) / 1024) * 1024;
    static constexpr int BAR_OFF = NS * STAGE;
    static constexpr int SMEM = BAR_OFF + 2 * NS * 8 + 1024;
};

struct GateParams {
    int T, H, dm;
    float eta_base;
    float *eta;
    int *status;
};

// byte offset of element (r, c) of a slice of 128-byte rows under the 128-byte swizzle
__device__ __forceinline__ uint32_t goff(int r, int c)
{
    const uint32_t a = static_cast<uint32_t>(r * 128 + c * 2);
    return a ^ (((a >> 7) & 7u) << 4);
}

template <int HP>
__global__ void __launch_bounds__(GateCfg<HP>::THREADS)
    ttt_eta_gate_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tth,
                        const GateParams p)
{
    using C = GateCfg<HP>;
    constexpr int NS = C::NS, NT = HP / 8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = 64 * blockIdx.x, b = blockIdx.y;
    const int nkc = (p.dm + 63) >> 6;
    const uint32_t full = base + C::BAR_OFF, empty = full + 8 * NS;
    if (threadIdx.x == 0) {
        prefetch_tmap(&tx);
        prefetch_tmap(&tth);
        for (int s = 0; s < NS; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 4);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == C::PW) {
        if (lane == 0) {
            int kc = 0;
            for (; kc < nkc; ++kc) {
                const int s = kc % NS;
                if (kc >= NS && !mbar_wait(empty + 8 * s, ((kc / NS) & 1) ^ 1, p.status, kSiteProducerEmpty))
                    break;
                const uint32_t st = base + s * C::STAGE;
                mbar_arrive_expect_tx(full + 8 * s, C::XB + HP * 128);
                tma_load_3d(st, &tx, full + 8 * s, 64 * kc, t0, b);
                tma_load_3d(st + C::XB, &tth, full + 8 * s, 64 * kc, 0, 0);
            }
            // the copies issued last land before the CTA can end
            for (int j = kc > NS ? kc - NS : 0; j < kc; ++j)
                if (!mbar_wait(full + 8 * (j % NS), (j / NS) & 1, p.status, kSiteDrain)) break;
        }
        return;
    }

    const int g = lane >> 2, t4 = lane & 3;
    const int rowA = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1), colA = 8 * (lane >> 4);
    const int rowB = (lane & 7) + 8 * (lane >> 4), colB = 8 * ((lane >> 3) & 1);
    float acc[NT][4] = {};
    for (int kc = 0; kc < nkc; ++kc) {
        const int s = kc % NS;
        if (!mbar_wait(full + 8 * s, (kc / NS) & 1, p.status, kSiteConsumerFull)) return;
        const uint32_t sx = base + s * C::STAGE, sth = sx + C::XB;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sx + goff(rowA, 16 * kk + colA), a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sth + goff(16 * np + rowB, 16 * kk + colB), b0, b1, b2, b3);
                mma_bf16(acc[2 * np], a0, a1, a2, a3, b0, b1);
                mma_bf16(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + 8 * s);
    }
    // accumulator (token 16 warp + g + 8 (i >> 1), head 8 nt + 2 t4 + (i & 1))
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = t0 + 16 * warp + g + 8 * (i >> 1), h = 8 * nt + 2 * t4 + (i & 1);
            if (t < p.T && h < p.H)
                p.eta[((size_t)b * p.H + h) * p.T + t] = p.eta_base / (1.f + expf(-acc[nt][i]));
        }
}

template <int HP>
int launch_gate_h(const GateArgs &a)
{
    using C = GateCfg<HP>;
    CUtensorMap mx, mth;
    // x as [B][T][dm] in boxes of 64 tokens x 64 features; theta as [1][H][dm] in
    // boxes of HP rows x 64 features (rows past H and features past dm read as zeros)
    if (!encode_token_map(&mx, a.x, a.B, a.T, a.dm, 64, 64) || !encode_token_map(&mth, a.theta, 1, a.H, a.dm, HP, 64))
        return -4;
    if (cudaFuncSetAttribute(ttt_eta_gate_kernel<HP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
        return -4;
    GateParams p;
    p.T = a.T;
    p.H = a.H;
    p.dm = a.dm;
    p.eta_base = a.eta_base;
    p.eta = a.eta;
    p.status = a.status;
    const dim3 grid((a.T + 63) / 64, a.B);
    ttt_eta_gate_kernel<HP><<<grid, C::THREADS, C::SMEM, a.stream>>>(mx, mth, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

int launch_eta_gate(const GateArgs &a)
{
    if (a.B == 0 || a.T == 0) return 0;
    if (a.H <= 16) return launch_gate_h<16>(a);
    if (a.H <= 32) return launch_gate_h<32>(a);
    if (a.H <= 64) return launch_gate_h<64>(a);
    return -2;
}

}  // namespace ttt
