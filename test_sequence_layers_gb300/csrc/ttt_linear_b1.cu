// ttt_linear_b1.cu -- TTT-Linear forward with mini-batches of one token (the delta
// rule), bf16 operands, fp32 state and arithmetic, d in {16, 32, 64, 128}.
//
// With b = 1 every token takes its gradient at the weights the previous token left
// ("Learning to (Learn at Test Time)", section 1.2.2: the mini-batch rule at b = 1;
// "Fast weights 与 TTT layers", section 1: the delta rule W_t = W_{t-1} +
// eta (v_t - W_{t-1} k_t) k_t^T in the column convention), so per token
//
//   e_t = k_t W - v_t,   W <- W - eta_t k_t^T e_t,   z_t = q_t W
//
// (the negative dot-product loss: e_t = -v_t).  Output column j of W evolves alone:
// e_t[j] = k_t . W[:, j] - v_t[j] and the update of W[:, j] reads e_t[j] only.  So
// the columns are spread over warps and CTAs, with no exchange between them: a warp
// holds two columns, sixteen lanes per column (eight when d = 16), each lane d/16
// entries of it; a token costs each lane a short dot product, a four-step shuffle
// reduction and d/16 fused multiply-adds (the output's dot product and reduction ride
// beside the next token's), and every SM sub-partition runs one warp.  Tokens arrive
// in 64-token blocks (k and q whole rows, v and z only the CTA's columns) by cp.async
// into two buffers, the next block's copies in flight during the current block; z is
// staged in shared memory and written once per block.
#include <cuda_bf16.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kB1TB = 64;  // tokens per block

// RG lanes per column (a reduction of log2 RG shuffles), 32 / RG columns per warp,
// up to four warps per CTA.  Measured on linear_125m_b1 (B1 H12 T2048 d64): 16 lanes
// per column 220 us, 8 lanes 267 us, 4 lanes 296 us, a whole warp (eight warps per
// CTA) 258 us.
template <int D>
struct B1Cfg {
    static constexpr int RG = D / 2 < 16 ? D / 2 : 16;
    static constexpr int R = D / RG;                         // rows of a column per lane
    static constexpr int CPW = 32 / RG;                      // columns per warp
    static constexpr int WARPS = D / CPW < 4 ? D / CPW : 4;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int COLS = CPW * WARPS;                 // output columns per CTA
    static constexpr int KQ = kB1TB * D * 2;                 // one block of k (or q) rows
    static constexpr int VZ = kB1TB * COLS * 2;              // one block of the CTA's v (or z) columns
    static constexpr int BUF = 2 * KQ + VZ + kB1TB * 4;      // k, q, v, eta of one block
    static constexpr int ZOFF = 2 * BUF;                     // two z staging tiles
    static constexpr int SMEM = ZOFF + 2 * VZ;
};

struct B1Params {
    int H, T, dot;
    const __nv_bfloat16 *q, *k, *v;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    __nv_bfloat16 *z;
    float *W_out;
};

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// R consecutive bf16 values at a 4-byte aligned shared address, as floats
template <int R>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *p, float (&f)[R])
{
    if constexpr (R % 8 == 0) {
#pragma unroll
        for (int i = 0; i < R / 8; ++i) {
            const uint4 u = reinterpret_cast<const uint4 *>(p)[i];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[8 * i + 2 * j] = bf16_lo(w[j]);
                f[8 * i + 2 * j + 1] = bf16_hi(w[j]);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < R / 2; ++j) {
            const uint32_t w = reinterpret_cast<const uint32_t *>(p)[j];
            f[2 * j] = bf16_lo(w);
            f[2 * j + 1] = bf16_hi(w);
        }
    }
}

template <int D>
__global__ void __launch_bounds__(B1Cfg<D>::THREADS) ttt_linear_b1_kernel(const B1Params p)
{
    using C = B1Cfg<D>;
    constexpr int R = C::R, RG = C::RG, COLS = C::COLS, THREADS = C::THREADS, NCT = D / COLS;
    extern __shared__ __align__(16) uint8_t smem[];
    const int bh = blockIdx.x / NCT, c0 = (blockIdx.x % NCT) * COLS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cj = lane / RG, rg = lane % RG;            // column of the warp, row group
    const int cl = C::CPW * warp + cj, col = c0 + cl;    // column inside the CTA / of W
    const int T = p.T, nblk = (T + kB1TB - 1) / kB1TB;
    const bool has_eta = p.eta != nullptr;
    const size_t tok0 = (size_t)bh * T;

    // the column's entries W[rg R + r][col]
    float w[R];
    {
        const float *W0 = p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * D * D;
#pragma unroll
        for (int r = 0; r < R; ++r) w[r] = W0[(size_t)(rg * R + r) * D + col];
    }

    // copies of block L into buffer L & 1 (rows past T are not copied, nor read)
    auto issue = [&](int L) {
        const uint32_t b = smem_u32(smem + (L & 1) * C::BUF);
        const int t0 = L * kB1TB, nt = min(kB1TB, T - t0);
        constexpr int RC = D / 8;  // 16-byte pieces of a k or q row
        for (int i = threadIdx.x; i < nt * RC; i += THREADS) {
            const int t = i / RC, c = i % RC;
            const size_t g = (tok0 + t0 + t) * D + 8 * c;
            cp_async_16(b + (t * D + 8 * c) * 2, p.k + g);
            cp_async_16(b + C::KQ + (t * D + 8 * c) * 2, p.q + g);
        }
        constexpr int VC = COLS / 8;  // 16-byte pieces of the CTA's v (or z) columns of a row
        for (int i = threadIdx.x; i < nt * VC; i += THREADS) {
            const int t = i / VC, c = i % VC;
            cp_async_16(b + 2 * C::KQ + (t * COLS + 8 * c) * 2, p.v + (tok0 + t0 + t) * D + c0 + 8 * c);
        }
        if (has_eta)
            for (int t = threadIdx.x; t < nt; t += THREADS)
                cp_async_4(b + 2 * C::KQ + C::VZ + 4 * t, p.eta + tok0 + t0 + t);
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    if (nblk > 0) issue(0);
    for (int L = 0; L < nblk; ++L) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();  // block L visible; every warp is done with block L - 1's buffers
        if (L + 1 < nblk) issue(L + 1);
        const uint8_t *buf = smem + (L & 1) * C::BUF;
        const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(buf) + rg * R;
        const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(buf + C::KQ) + rg * R;
        const __nv_bfloat16 *vs = reinterpret_cast<const __nv_bfloat16 *>(buf + 2 * C::KQ) + cl;
        const float *es = reinterpret_cast<const float *>(buf + 2 * C::KQ + C::VZ);
        __nv_bfloat16 *zs = reinterpret_cast<__nv_bfloat16 *>(smem + C::ZOFF + (L & 1) * C::VZ) + cl;
        const int t0 = L * kB1TB, nt = min(kB1TB, T - t0);
        // z_t = q_t W_t (token t's own write included) reads the weights that token
        // t + 1's residual reads, so the two dot products and their reductions are
        // formed side by side, one token apart: the output's shuffles run in the
        // shadow of the state chain's
        float qp[R];  // q of the previous token
        auto dot2 = [&](const float (&x)[R]) {
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int r = 0; r < R; r += 2) {
                d0 = fmaf(x[r], w[r], d0);
                d1 = fmaf(x[r + 1], w[r + 1], d1);
            }
            return d0 + d1;
        };
        load_row<R>(qs, qp);
#pragma unroll 2
        for (int t = 0; t < nt; ++t) {
            float kf[R];
            load_row<R>(ks + t * D, kf);
            const float vt = __bfloat162float(vs[t * COLS]);
            const float et = has_eta ? es[t] : p.eta_scalar;
            // e_t = k_t . W[:, col] - v_t[col] (dot loss: -v_t), reduced over the
            // column's eight lanes together with the previous token's output
            float a = p.dot ? 0.f : dot2(kf);
            float zz = t > 0 ? dot2(qp) : 0.f;
#pragma unroll
            for (int m = 1; m < RG; m <<= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, m);
                zz += __shfl_xor_sync(0xffffffffu, zz, m);
            }
            const float s = -et * (a - vt);
#pragma unroll
            for (int r = 0; r < R; ++r) w[r] = fmaf(s, kf[r], w[r]);
            if (t > 0 && rg == 0) zs[(t - 1) * COLS] = __float2bfloat16_rn(zz);
            load_row<R>(qs + t * D, qp);
        }
        {  // the block's last output
            float zz = dot2(qp);
#pragma unroll
            for (int m = 1; m < RG; m <<= 1) zz += __shfl_xor_sync(0xffffffffu, zz, m);
            if (rg == 0) zs[(nt - 1) * COLS] = __float2bfloat16_rn(zz);
        }
        __syncthreads();  // the block's z tile is complete
        {
            const uint32_t *zt = reinterpret_cast<const uint32_t *>(smem + C::ZOFF + (L & 1) * C::VZ);
            constexpr int VC = COLS / 8;
            for (int i = threadIdx.x; i < nt * VC; i += THREADS) {
                const int t = i / VC, c = i % VC;
                const uint4 u = reinterpret_cast<const uint4 *>(zt)[t * VC + c];
                *reinterpret_cast<uint4 *>(p.z + (tok0 + t0 + t) * D + c0 + 8 * c) = u;
            }
        }
    }
    if (p.W_out) {
        float *Wo = p.W_out + (size_t)bh * D * D;
#pragma unroll
        for (int r = 0; r < R; ++r) Wo[(size_t)(rg * R + r) * D + col] = w[r];
    }
}

template <int D>
int launch_b1_t(const LinearArgs &a)
{
    using C = B1Cfg<D>;
    if (cudaFuncSetAttribute(ttt_linear_b1_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
        return -4;
    B1Params p;
    p.H = a.H;
    p.T = a.T;
    p.dot = a.loss;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k = static_cast<const __nv_bfloat16 *>(a.k);
    p.v = static_cast<const __nv_bfloat16 *>(a.v);
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W0 = a.W0;
    p.w0_bstride = a.w0_bstride;
    p.z = static_cast<__nv_bfloat16 *>(a.z);
    p.W_out = a.W_out;
    ttt_linear_b1_kernel<D><<<a.B * a.H * (D / C::COLS), C::THREADS, C::SMEM, a.stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

// b = 1, bf16, one inner epoch, no inner norm, d in {16, 32, 64, 128}; -2 otherwise.
int launch_linear_b1(const LinearArgs &a)
{
    if (a.b != 1 || a.epochs != 1 || a.ln_gamma) return -2;
    if (a.B * a.H == 0) return 0;
    switch (a.d) {
    case 16: return launch_b1_t<16>(a);
    case 32: return launch_b1_t<32>(a);
    case 64: return launch_b1_t<64>(a);
    case 128: return launch_b1_t<128>(a);
    default: return -2;
    }
}

}  // namespace ttt
