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
// per-thread partial sums are reduced through shared memory.  K (then Q) sits in
// shared memory as fp32 in a zero-bordered grid, so the taps need no bounds tests,
// and each thread walks whole rows with a 3 x 3 register window (three new taps per
// position instead of nine).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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

// shared memory: a zero-bordered (height+2) x (width+2) grid of fp32 tokens
// (K, then Q), V [N][d] in the I/O type, taps W [9][d], eta [N], partial tap
// gradients [parts][9][d]
__host__ __device__ inline size_t dw_smem_bytes(int hh, int ww, int d, int es)
{
    const int parts = kDwThreads / (d / 2);
    return 4 * (size_t)(hh + 2) * (ww + 2) * d + (size_t)hh * ww * d * es +
           4 * (9 * (size_t)d + (size_t)hh * ww + (size_t)parts * 9 * d);
}

// The tokens of one sequence into the interior of the padded fp32 grid (the border
// is left as it is).  Every thread first issues all of its 16-byte loads, then
// converts and stores, so the loads of a thread are in flight together.
template <typename TIO>
__device__ __forceinline__ void stage_grid(float *grid, const TIO *src, int hh, int ww, int d)
{
    constexpr int EPV = 16 / sizeof(TIO);  // elements per 16-byte vector
    const int nvec = hh * ww * d / EPV, vpr = d / EPV;  // vectors in all / per token
    constexpr int U = 8;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += U * kDwThreads) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kDwThreads;
            if (v < nvec) buf[u] = reinterpret_cast<const uint4 *>(src)[v];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * kDwThreads;
            if (v >= nvec) break;
            const int tok = v / vpr, c = (v - tok * vpr) * EPV;
            const int y = tok / ww, x = tok - y * ww;
            float *dst = grid + ((size_t)(y + 1) * (ww + 2) + x + 1) * d + c;
            if constexpr (sizeof(TIO) == 2) {
                const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&buf[u]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(h[i]);
                    dst[2 * i] = f.x;
                    dst[2 * i + 1] = f.y;
                }
            } else {
                *reinterpret_cast<uint4 *>(dst) = buf[u];
            }
        }
    }
}

template <typename TIO>
__device__ __forceinline__ void stage_flat(TIO *dst, const TIO *src, int n_elem)
{
    const int nv = n_elem * (int)sizeof(TIO) / 16;
    constexpr int U = 8;
    for (int v0 = threadIdx.x; v0 < nv; v0 += U * kDwThreads) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + u * kDwThreads < nv) buf[u] = reinterpret_cast<const uint4 *>(src)[v0 + u * kDwThreads];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + u * kDwThreads < nv) reinterpret_cast<uint4 *>(dst)[v0 + u * kDwThreads] = buf[u];
    }
}

template <typename TIO>
__global__ void __launch_bounds__(kDwThreads) ttt_dwconv_kernel(const DwParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int d = p.d, hh = p.hh, ww = p.ww, N = hh * ww, gw = ww + 2;
    float *sG = reinterpret_cast<float *>(smem);                 // padded grid: K, then Q
    TIO *sV = reinterpret_cast<TIO *>(sG + (size_t)(hh + 2) * gw * d);
    float *sW = reinterpret_cast<float *>(sV + (size_t)N * d);
    float *sEta = sW + 9 * d;
    float *sPart = sEta + N;
    const int bh = blockIdx.x, tid = threadIdx.x;
    const int npair = d / 2, parts = kDwThreads / npair;
    const int cp = tid % npair, part = tid / npair, c = 2 * cp;
    const size_t off = (size_t)bh * N * d;

    // zero border of the grid (rows 0 and hh+1, columns 0 and ww+1)
    for (int i = tid; i < 2 * (gw + hh) * d; i += kDwThreads) {
        const int cell = i / d, cc = i - cell * d;
        int y, x;
        if (cell < gw) { y = 0; x = cell; }
        else if (cell < 2 * gw) { y = hh + 1; x = cell - gw; }
        else { const int r = cell - 2 * gw; y = 1 + (r >> 1); x = (r & 1) ? ww + 1 : 0; }
        sG[((size_t)y * gw + x) * d + cc] = 0.f;
    }
    stage_grid(sG, static_cast<const TIO *>(p.k) + off, hh, ww, d);
    stage_flat(sV, static_cast<const TIO *>(p.v) + off, N * d);
    const float *W0 = p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * 9 * d;
    for (int i = tid; i < 9 * d; i += kDwThreads) sW[i] = W0[i];
    for (int i = tid; i < N; i += kDwThreads) sEta[i] = p.eta ? p.eta[(size_t)bh * N + i] : p.eta_scalar;
    __syncthreads();

    const bool active = tid < parts * npair;
    // taps of grid cell (y, x) of the padded grid for this thread's channel pair
    auto tap = [&](int y, int x) { return *reinterpret_cast<const float2 *>(sG + ((size_t)y * gw + x) * d + c); };

    for (int ep = 0; ep < p.epochs; ++ep) {
        float w[9][2], g[9][2];
#pragma unroll
        for (int o = 0; o < 9; ++o) {
            w[o][0] = sW[o * d + c];
            w[o][1] = sW[o * d + c + 1];
            g[o][0] = g[o][1] = 0.f;
        }
        if (active) {
            for (int y = part; y < hh; y += parts) {
                // sliding 3 x 3 window over padded rows y .. y+2; column j of the
                // window holds padded column x + j for output column x
                float2 win[3][3];
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    win[r][0] = tap(y + r, 0);
                    win[r][1] = tap(y + r, 1);
                }
                for (int x = 0; x < ww; ++x) {
#pragma unroll
                    for (int r = 0; r < 3; ++r) win[r][2] = tap(y + r, x + 2);
                    const int pos = y * ww + x;
                    const float2 vv = ld2(sV + (size_t)pos * d + c);
                    float e0 = -vv.x, e1 = -vv.y;
                    if (!p.dot) {
#pragma unroll
                        for (int o = 0; o < 9; ++o) {
                            e0 = fmaf(win[o / 3][o % 3].x, w[o][0], e0);
                            e1 = fmaf(win[o / 3][o % 3].y, w[o][1], e1);
                        }
                    }
                    const float et = sEta[pos];
                    e0 *= et;
                    e1 *= et;
#pragma unroll
                    for (int o = 0; o < 9; ++o) {
                        g[o][0] = fmaf(e0, win[o / 3][o % 3].x, g[o][0]);
                        g[o][1] = fmaf(e1, win[o / 3][o % 3].y, g[o][1]);
                    }
#pragma unroll
                    for (int r = 0; r < 3; ++r) {
                        win[r][0] = win[r][1];
                        win[r][1] = win[r][2];
                    }
                }
            }
#pragma unroll
            for (int o = 0; o < 9; ++o) {
                sPart[((size_t)part * 9 + o) * d + c] = g[o][0];
                sPart[((size_t)part * 9 + o) * d + c + 1] = g[o][1];
            }
        }
        __syncthreads();  // partial sums visible; every read of sW is done
        for (int i = tid; i < 9 * d; i += kDwThreads) {
            float s = 0.f;
            for (int r = 0; r < parts; ++r) s += sPart[(size_t)r * 9 * d + i];
            sW[i] -= s;
        }
        __syncthreads();  // the epoch's taps visible; every read of the grid is done
    }

    // output pass: Q in K's place (the border stays zero)
    stage_grid(sG, static_cast<const TIO *>(p.q) + off, hh, ww, d);
    __syncthreads();
    if (active) {
        float w[9][2];
#pragma unroll
        for (int o = 0; o < 9; ++o) {
            w[o][0] = sW[o * d + c];
            w[o][1] = sW[o * d + c + 1];
        }
        TIO *z = static_cast<TIO *>(p.z) + off;
        for (int y = part; y < hh; y += parts) {
            float2 win[3][3];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                win[r][0] = tap(y + r, 0);
                win[r][1] = tap(y + r, 1);
            }
            for (int x = 0; x < ww; ++x) {
#pragma unroll
                for (int r = 0; r < 3; ++r) win[r][2] = tap(y + r, x + 2);
                float z0 = 0.f, z1 = 0.f;
#pragma unroll
                for (int o = 0; o < 9; ++o) {
                    z0 = fmaf(win[o / 3][o % 3].x, w[o][0], z0);
                    z1 = fmaf(win[o / 3][o % 3].y, w[o][1], z1);
                }
                st2(z + (size_t)(y * ww + x) * d + c, z0, z1);
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    win[r][0] = win[r][1];
                    win[r][1] = win[r][2];
                }
            }
        }
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
