// ttt_dwconv.cu -- TTT with a depthwise 3x3 convolution as the inner model (the
// ViT3 article, observation 6: the inner model of vision TTT can be a small
// convolution, whose taps absorb the keys' and values' global information while
// the query pass keeps the kernel's local receptive field; the ViT3 block uses a
// depthwise one).  Full-batch inner gradient descent over the N = height * width
// tokens of a sequence (observation 2), one or more epochs, every query reading
// the final taps.
//
// The tokens are the pixels of a height x width grid in row-major order and
//     f(X; W)[p][c] = sum_{o in 3x3} X[p + o][c] * W[o][c]
// (cross-correlation, zero outside the grid).  One epoch at start taps Ws:
//     e[p][c] = f(K; Ws)[p][c] - V[p][c]        (MSE; the dot loss has e = -V)
//     W[o][c] -= sum_p eta_p e[p][c] K[p + o][c]
// and the output is Z = f(Q; W_final).  Nothing here is a contraction over a
// shared dimension (each channel has its own nine taps), so the work runs on the
// CUDA cores: one CTA per (batch, head) holds K and V in shared memory in the I/O
// type; each thread owns a pair of channels and a stride of positions, forms each
// residual on the fly and accumulates the nine tap gradients in registers; the
// per-thread partial sums are reduced through shared memory.  K and Q sit in
// shared memory in zero-bordered grids (I/O type), so the taps need no bounds
// tests; each thread walks whole rows with a 3 x 3 register window (three new taps
// per position instead of nine).  All of a sequence's token copies (K, V, then Q)
// are issued at the start as bulk asynchronous copies (one per grid row), so Q lands
// while the epochs run; channel pairs use the paired fp32 FMA.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

constexpr int kDwThreads = 256;

struct DwParams {
    int H, hh, ww, d, dot, epochs;
    const void *q, *k, *v;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    void *z;
    float *W_out;
    int *status;
};

template <typename TIO>
__device__ __forceinline__ float2 ld2(const TIO *p)
{
    if constexpr (sizeof(TIO) == 2) {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(p);
        return __bfloat1622float2(v);
    } else {
        return *reinterpret_cast<const float2 *>(p);
    }
}

template <typename TIO>
__device__ __forceinline__ void st2(TIO *p, float a, float b)
{
    if constexpr (sizeof(TIO) == 2)
        *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
    else
        *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}

// shared memory: two mbarriers, two zero-bordered (height+2) x (width+2) token
// grids in the I/O type (K, Q), V [N][d], taps W [9][d], partial tap gradients
// [parts][9][d] (paired 8-byte accesses, so ahead of the odd-length eta), eta [N]
__host__ __device__ inline size_t dw_smem_bytes(int hh, int ww, int d, int es)
{
    const int parts = kDwThreads / (d / 2);
    return 16 + 2 * (size_t)(hh + 2) * (ww + 2) * d * es + (size_t)hh * ww * d * es +
           4 * (9 * (size_t)d + (size_t)hh * ww + (size_t)parts * 9 * d);
}

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes a multiple of
// 16), completion counted on the mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// zero border (rows 0 and hh+1, columns 0 and ww+1) of a padded grid, in 16-byte
// pieces (a cell is d * sizeof(TIO) bytes, a multiple of 16)
template <typename TIO>
__device__ __forceinline__ void zero_border(TIO *grid, int hh, int ww, int d)
{
    const int gw = ww + 2, vpc = d * (int)sizeof(TIO) / 16;
    uint4 *g4 = reinterpret_cast<uint4 *>(grid);
    for (int i = threadIdx.x; i < 2 * (gw + hh) * vpc; i += kDwThreads) {
        const int cell = i / vpc, piece = i - cell * vpc;
        int y, x;
        if (cell < gw) { y = 0; x = cell; }
        else if (cell < 2 * gw) { y = hh + 1; x = cell - gw; }
        else { const int r = cell - 2 * gw; y = 1 + (r >> 1); x = (r & 1) ? ww + 1 : 0; }
        g4[((size_t)y * gw + x) * vpc + piece] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Walks the positions p0 .. p1-1 (row-major) of a padded grid with a 3 x 3 window
// for channel pair c, one row segment at a time.  The window's columns rotate
// through three register triples (unrolled by three, so no moves);
// step(pos, a, b, n) gets the padded columns x, x+1, x+2 of padded rows y .. y+2
// for output (y, x) = pos, i.e. tap (r, j) is {a, b, n}[j][r].
template <typename TIO, typename Step>
__device__ __forceinline__ void walk_run(const TIO *g, int p0, int p1, int ww, int d, int c, Step &&step)
{
    const int gw = ww + 2;
    int y = p0 < p1 ? p0 / ww : 0, x0 = p0 - y * ww;  // (ww > 0 whenever the run is not empty)
    while (p0 < p1) {
        const int x1 = min(ww, x0 + (p1 - p0)), base = y * ww;
        float2 A[3], B[3], C[3];
        auto col = [&](int xc, float2 (&cc)[3]) {
#pragma unroll
            for (int r = 0; r < 3; ++r) cc[r] = ld2(g + ((size_t)(y + r) * gw + xc) * d + c);
        };
        col(x0, A);
        col(x0 + 1, B);
        int x = x0;
        for (; x + 3 <= x1; x += 3) {
            col(x + 2, C);
            step(base + x, A, B, C);
            col(x + 3, A);
            step(base + x + 1, B, C, A);
            col(x + 4, B);
            step(base + x + 2, C, A, B);
        }
        if (x < x1) {
            col(x + 2, C);
            step(base + x, A, B, C);
            if (x + 1 < x1) {
                col(x + 3, A);
                step(base + x + 1, B, C, A);
            }
        }
        p0 += x1 - x0;
        ++y;
        x0 = 0;
    }
}

// One epoch's partial tap gradients of this thread's channel pair over its run:
// g[o] += s_p e_p K[p + o], with e_p = f(K; W)_p - V_p (MSE) or V_p (DOT, whose
// true residual -V_p has its sign applied in the update), s_p = eta_p (ETA) or 1
// (a scalar eta is applied in the update).
template <typename TIO, bool DOT, bool ETA>
__device__ __forceinline__ void epoch_grad(const TIO *sK, const TIO *sV, const float *sEta, const float2 (&w)[9],
                                           float2 (&g)[9], int p0, int p1, int ww, int d, int c)
{
    walk_run(sK, p0, p1, ww, d, c, [&](int pos, const float2(&a)[3], const float2(&b)[3], const float2(&n)[3]) {
        const float2 vv = ld2(sV + (size_t)pos * d + c);
        float2 e;
        if constexpr (DOT) {
            e = vv;
        } else {
            e = make_float2(-vv.x, -vv.y);
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                e = fma2(a[r], w[3 * r], e);
                e = fma2(b[r], w[3 * r + 1], e);
                e = fma2(n[r], w[3 * r + 2], e);
            }
        }
        if constexpr (ETA) {
            const float et = sEta[pos];
            e = __fmul2_rn(e, make_float2(et, et));
        }
#pragma unroll
        for (int r = 0; r < 3; ++r) {
            g[3 * r] = fma2(e, a[r], g[3 * r]);
            g[3 * r + 1] = fma2(e, b[r], g[3 * r + 1]);
            g[3 * r + 2] = fma2(e, n[r], g[3 * r + 2]);
        }
    });
}

template <typename TIO>
__global__ void __launch_bounds__(kDwThreads) ttt_dwconv_kernel(const DwParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int d = p.d, hh = p.hh, ww = p.ww, N = hh * ww, gw = ww + 2;
    const size_t gsz = (size_t)(hh + 2) * gw * d;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // [0]: K and V, [1]: Q
    TIO *sK = reinterpret_cast<TIO *>(smem + 16);         // padded grid of K
    TIO *sQ = sK + gsz;                                   // padded grid of Q
    TIO *sV = sQ + gsz;                                   // V [N][d]
    float *sW = reinterpret_cast<float *>(sV + (size_t)N * d);  // 16-byte aligned
    float *sPart = sW + 9 * d;                                   // 8-byte aligned (d % 8 == 0)
    float *sEta = sPart + (size_t)(kDwThreads / (d / 2)) * 9 * d;
    const int bh = blockIdx.x, tid = threadIdx.x;
    const int npair = d / 2, parts = kDwThreads / npair;
    const int part = tid / npair, c = 2 * (tid % npair);
    const size_t off = (size_t)bh * N * d;
    const uint32_t bar_kv = smem_u32(bars), bar_q = smem_u32(bars + 1);

    if (tid == 0) {
        mbar_init(bar_kv, 1);
        mbar_init(bar_q, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // warp 0 issues every token copy at once, one bulk copy per grid row (the
    // interior of a padded row is contiguous) and one for V: K and V complete on
    // bar_kv, Q on bar_q, so Q lands while the epochs run
    if (tid < 32) {
        const uint32_t row = (uint32_t)(ww * d * sizeof(TIO));
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_kv, 2u * (uint32_t)hh * row);
            mbar_arrive_expect_tx(bar_q, (uint32_t)hh * row);
        }
        __syncwarp();
        if (N > 0) {
            const TIO *gk = static_cast<const TIO *>(p.k) + off, *gq = static_cast<const TIO *>(p.q) + off;
            for (int y = tid; y < hh; y += 32) {
                const uint32_t o = (uint32_t)(((size_t)(y + 1) * gw + 1) * d * sizeof(TIO));
                bulk_load(smem_u32(sK) + o, gk + (size_t)y * ww * d, row, bar_kv);
                bulk_load(smem_u32(sQ) + o, gq + (size_t)y * ww * d, row, bar_q);
            }
            if (tid == 0) bulk_load(smem_u32(sV), static_cast<const TIO *>(p.v) + off, (uint32_t)hh * row, bar_kv);
        }
    }
    zero_border(sK, hh, ww, d);
    zero_border(sQ, hh, ww, d);
    const float *W0 = p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * 9 * d;
    for (int i = tid; i < 9 * d; i += kDwThreads) sW[i] = W0[i];
    if (p.eta)
        for (int i = tid; i < N; i += kDwThreads) sEta[i] = p.eta[(size_t)bh * N + i];
    // K and V landed (every thread observes the barrier) and the generic stores
    // above are visible; a timeout (never expected) is CTA-uniform after the vote
    if (!__syncthreads_and(mbar_wait(bar_kv, 0, p.status, kSiteStage))) {
        mbar_wait(bar_q, 0, p.status, kSiteStage);
        return;
    }

    const bool active = tid < parts * npair;
    // this thread's run of positions: an even share of the N in row-major order
    const int p0 = (int)((long long)N * part / parts), p1 = (int)((long long)N * (part + 1) / parts);
    // W -= upd * (summed partials): the dot loss's sign and a scalar eta
    const float upd = (p.dot ? -1.f : 1.f) * (p.eta ? 1.f : p.eta_scalar);
    for (int ep = 0; ep < p.epochs; ++ep) {
        if (active) {
            float2 w[9], g[9];
#pragma unroll
            for (int o = 0; o < 9; ++o) {
                w[o] = *reinterpret_cast<const float2 *>(sW + o * d + c);
                g[o] = make_float2(0.f, 0.f);
            }
            if (p.dot) {
                if (p.eta) epoch_grad<TIO, true, true>(sK, sV, sEta, w, g, p0, p1, ww, d, c);
                else epoch_grad<TIO, true, false>(sK, sV, sEta, w, g, p0, p1, ww, d, c);
            } else {
                if (p.eta) epoch_grad<TIO, false, true>(sK, sV, sEta, w, g, p0, p1, ww, d, c);
                else epoch_grad<TIO, false, false>(sK, sV, sEta, w, g, p0, p1, ww, d, c);
            }
#pragma unroll
            for (int o = 0; o < 9; ++o) *reinterpret_cast<float2 *>(sPart + ((size_t)part * 9 + o) * d + c) = g[o];
        }
        __syncthreads();  // partial sums visible; every read of sW is done
        for (int i = tid; i < 9 * d; i += kDwThreads) {
            float s = 0.f;
            for (int r = 0; r < parts; ++r) s += sPart[(size_t)r * 9 * d + i];
            sW[i] = fmaf(-upd, s, sW[i]);
        }
        __syncthreads();  // the epoch's taps visible
    }

    // output pass over the Q grid
    if (!__syncthreads_and(mbar_wait(bar_q, 0, p.status, kSiteStage))) return;
    if (active) {
        float2 w[9];
#pragma unroll
        for (int o = 0; o < 9; ++o) w[o] = *reinterpret_cast<const float2 *>(sW + o * d + c);
        TIO *z = static_cast<TIO *>(p.z) + off;
        walk_run(sQ, p0, p1, ww, d, c, [&](int pos, const float2(&a)[3], const float2(&b)[3], const float2(&n)[3]) {
            float2 zz = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                zz = fma2(a[r], w[3 * r], zz);
                zz = fma2(b[r], w[3 * r + 1], zz);
                zz = fma2(n[r], w[3 * r + 2], zz);
            }
            st2(z + (size_t)pos * d + c, zz.x, zz.y);
        });
    }
    if (p.W_out)
        for (int i = tid; i < 9 * d; i += kDwThreads) p.W_out[(size_t)bh * 9 * d + i] = sW[i];
}

}  // namespace

size_t dwconv_smem(int hh, int ww, int d, int es) { return dw_smem_bytes(hh, ww, d, es); }

int launch_dwconv(const DwconvArgs &a)
{
    const int es = a.bf16 ? 2 : 4;
    const size_t smem = dw_smem_bytes(a.hh, a.ww, a.d, es);
    DwParams p;
    p.H = a.H;
    p.hh = a.hh;
    p.ww = a.ww;
    p.d = a.d;
    p.dot = a.loss;
    p.epochs = a.epochs;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W0 = a.W0;
    p.w0_bstride = a.w0_bstride;
    p.z = a.z;
    p.W_out = a.W_out;
    p.status = a.status;
    if (a.bf16) {
        if (cudaFuncSetAttribute(ttt_dwconv_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return -4;
        ttt_dwconv_kernel<__nv_bfloat16><<<a.B * a.H, kDwThreads, smem, a.stream>>>(p);
    } else {
        if (cudaFuncSetAttribute(ttt_dwconv_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return -4;
        ttt_dwconv_kernel<float><<<a.B * a.H, kDwThreads, smem, a.stream>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace ttt
