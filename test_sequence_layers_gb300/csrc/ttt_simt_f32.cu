// ttt_simt_f32.cu -- fp32 CUDA-core paths of the TTT layer forward (fp32 I/O).
//
// These keep every operand in fp32 (no bf16, no TF32), for callers that need the
// fp32 accuracy class.  One CTA per (batch, head) chain holds the inner weights in
// shared memory and walks the tokens in order: every token of a mini-batch takes
// its gradient at the block's start weights (kept as a copy), and the running
// weights receive each token's write before its query reads them (causal) or
// after the whole block (non-causal) -- the mini-batch rule of the "Learning to
// (Learn at Test Time)" walkthrough, section 1.2.2, evaluated directly.
#include <cuda_runtime.h>

#include "ttt_internal.h"

namespace ttt {

namespace {

constexpr int kThreads = 256;
// Tokens whose k, v, q and eta are copied into shared memory together: one round trip
// to memory per tile instead of one per token on the serial path.
constexpr int kTile = 32;

struct LinF32Params {
    int H, T, d, b, causal, dot, epochs;  // dot: negative dot-product loss; epochs: passes per block
    const float *ln_gamma, *ln_beta;      // inner norm f(x) = x + LN(x W), [H][d] (or null)
    float ln_eps;
    const float *q, *k, *v, *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    float *z, *W_out;
};

// mean and 1 / sqrt(var + eps) of the D values x (every calling thread reads all)
__device__ __forceinline__ void row_stats(const float *x, int D, float eps, float &mu, float &rs)
{
    float s = 0.f, s2 = 0.f;
    for (int i = 0; i < D; ++i) s += x[i];
    mu = s / D;
    for (int i = 0; i < D; ++i) s2 += (x[i] - mu) * (x[i] - mu);
    rs = rsqrtf(s2 / D + eps);
}

// z = q + LN(y) for the row y (threads tid < D; y already in shared memory)
__device__ __forceinline__ float ln_out(const LinF32Params &p, const float *gm, const float *bt, const float *y,
                                        const float *qq, int D, int tid)
{
    float mu, rs;
    row_stats(y, D, p.ln_eps, mu, rs);
    return qq[tid] + fmaf(gm[tid], (y[tid] - mu) * rs, bt[tid]);
}

__global__ void __launch_bounds__(kThreads) ttt_linear_f32_kernel(const LinF32Params p)
{
    extern __shared__ float sm[];
    const int D = p.d, T = p.T, tid = threadIdx.x;
    float *W = sm, *Ws = W + D * D, *ee = Ws + D * D;
    float *yh = ee + D, *gs = yh + D;  // inner norm scratch
    float *kt = gs + D, *vt = kt + kTile * D, *qt = vt + kTile * D, *et = qt + kTile * D;  // token tile
    const bool ln = p.ln_gamma != nullptr;
    const float *gm = ln ? p.ln_gamma + (size_t)(blockIdx.x % p.H) * D : nullptr;
    const float *bt = ln ? p.ln_beta + (size_t)(blockIdx.x % p.H) * D : nullptr;
    const int bh = blockIdx.x;
    const float *W0 = p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * D * D;
    for (int i = tid; i < D * D; i += blockDim.x) W[i] = W0[i];
    const float *q = p.q + (size_t)bh * T * D, *k = p.k + (size_t)bh * T * D;
    const float *v = p.v + (size_t)bh * T * D;
    float *z = p.z + (size_t)bh * T * D;
    // tokens [t0, t1) into the tile (q alone for the non-causal output pass)
    auto load_tile = [&](int t0, int t1, bool q_only) {
        __syncthreads();  // the previous tile's readers are done
        const int n = (t1 - t0) * D;
        for (int i = tid; i < n; i += blockDim.x) {
            qt[i] = q[(size_t)t0 * D + i];
            if (!q_only) {
                kt[i] = k[(size_t)t0 * D + i];
                vt[i] = v[(size_t)t0 * D + i];
            }
        }
        if (!q_only)
            for (int i = tid; i < t1 - t0; i += blockDim.x) et[i] = p.eta ? p.eta[(size_t)bh * T + t0 + i] : p.eta_scalar;
        __syncthreads();
    };

    for (int n0 = 0; n0 < T; n0 += p.b) {
        const int n1 = min(n0 + p.b, T);
        for (int ep = 0; ep < p.epochs; ++ep) {  // more than one only for one non-causal block
        __syncthreads();
        for (int i = tid; i < D * D; i += blockDim.x) Ws[i] = W[i];
        for (int t = n0; t < n1; ++t) {
            if ((t - n0) % kTile == 0) load_tile(t, min(n1, t + kTile), false);
            const int ti = (t - n0) % kTile;
            const float *kk = kt + ti * D, *vv = vt + ti * D, *qq = qt + ti * D;
            __syncthreads();  // the previous token's readers of ee and W are done
            if (tid < D) {  // e = k_t W_start - v_t (dot loss: e = -v_t; norm: y = k_t W_start)
                float s = 0.f;
                if (!p.dot)
                    for (int i = 0; i < D; ++i) s = fmaf(kk[i], Ws[i * D + tid], s);
                ee[tid] = ln ? s : s - vv[tid];
            }
            __syncthreads();
            if (ln) {  // gradient through x + LN(y): dy = (g - mean g - yh mean(g yh)) / s, g = gamma e
                float mu = 0.f, rs = 0.f;
                if (tid < D) {
                    row_stats(ee, D, p.ln_eps, mu, rs);
                    yh[tid] = (ee[tid] - mu) * rs;
                    gs[tid] = gm[tid] * (kk[tid] + fmaf(gm[tid], yh[tid], bt[tid]) - vv[tid]);
                }
                __syncthreads();
                if (tid < D) {
                    float mg = 0.f, mgy = 0.f;
                    for (int i = 0; i < D; ++i) {
                        mg += gs[i];
                        mgy += gs[i] * yh[i];
                    }
                    ee[tid] = (gs[tid] - mg / D - yh[tid] * (mgy / D)) * rs;
                }
                __syncthreads();
            }
            const float eta_t = et[ti];
            for (int i = tid; i < D * D; i += blockDim.x)  // W -= eta k_t^T e
                W[i] = fmaf(-eta_t * kk[i / D], ee[i % D], W[i]);
            if (p.causal) {
                __syncthreads();
                float s = 0.f;
                if (tid < D) {
                    for (int i = 0; i < D; ++i) s = fmaf(qq[i], W[i * D + tid], s);
                    if (ln) yh[tid] = s;
                }
                if (ln) {
                    __syncthreads();
                    if (tid < D) s = ln_out(p, gm, bt, yh, qq, D, tid);
                }
                if (tid < D) z[(size_t)t * D + tid] = s;
            }
        }
        }  // epochs
        if (!p.causal) {
            for (int t = n0; t < n1; ++t) {
                if ((t - n0) % kTile == 0) load_tile(t, min(n1, t + kTile), true);
                const float *qq = qt + ((t - n0) % kTile) * D;
                __syncthreads();
                float s = 0.f;
                if (tid < D) {
                    for (int i = 0; i < D; ++i) s = fmaf(qq[i], W[i * D + tid], s);
                    if (ln) yh[tid] = s;
                }
                if (ln) {
                    __syncthreads();
                    if (tid < D) s = ln_out(p, gm, bt, yh, qq, D, tid);
                }
                if (tid < D) z[(size_t)t * D + tid] = s;
            }
        }
    }
    __syncthreads();
    if (p.W_out)
        for (int i = tid; i < D * D; i += blockDim.x) p.W_out[(size_t)bh * D * D + i] = W[i];
}

}  // namespace

int launch_linear_f32(const LinearArgs &a)
{
    const int D = a.d;
    const size_t smem = sizeof(float) * (2 * D * D + 3 * D + kTile * (3 * D + 1));
    if (cudaFuncSetAttribute(ttt_linear_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return -4;
    LinF32Params p;
    p.H = a.H;
    p.T = a.T;
    p.d = D;
    p.b = a.b;
    p.causal = a.causal;
    p.dot = a.loss;
    p.epochs = a.epochs;
    p.ln_gamma = a.ln_gamma;
    p.ln_beta = a.ln_beta;
    p.ln_eps = a.ln_eps;
    p.q = static_cast<const float *>(a.q);
    p.k = static_cast<const float *>(a.k);
    p.v = static_cast<const float *>(a.v);
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W0 = a.W0;
    p.w0_bstride = a.w0_bstride;
    p.z = static_cast<float *>(a.z);
    p.W_out = a.W_out;
    ttt_linear_f32_kernel<<<a.B * a.H, kThreads, smem, a.stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}


namespace {

struct MlpF32Params {
    int H, T, d, m, b, causal, per_batch, act;  // act: 0 SiLU, 1 GELU (h Phi(h), erf form)
    const float *ln_gamma, *ln_beta;             // inner norm x + LN(mlp(x)), [H][d] (or null)
    float ln_eps;
    const float *q, *k, *v, *eta;
    float eta_scalar;
    const float *W1, *c1, *W2, *c2;
    float *z, *W1o, *c1o, *W2o, *c2o;
};

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }

// act(h) and act'(h) of the inner MLP
__device__ __forceinline__ float act_f32(int act, float h)
{
    return act ? h * (0.5f + 0.5f * erff(h * 0.70710678118654752f)) : h * sigmoidf_(h);
}

__device__ __forceinline__ float act_d_f32(int act, float h)
{
    if (act) {
        const float Phi = 0.5f + 0.5f * erff(h * 0.70710678118654752f);
        return Phi + h * 0.39894228040143268f * expf(-0.5f * h * h);
    }
    const float sg = sigmoidf_(h);
    return sg * (1.f + h * (1.f - sg));
}

// floats of shared memory used by the fp32 MLP kernel
__host__ __device__ inline size_t mlp_f32_floats(int d, int m)
{
    return 2 * ((size_t)d * m + m + (size_t)m * d + d) + 4 * (size_t)m + 5 * (size_t)d;
}

// mean and 1 / sqrt(var + eps) of the n values x (every calling thread reads all)
__device__ __forceinline__ void row_stats_f32(const float *x, int n, float eps, float &mu, float &rs)
{
    float s = 0.f, s2 = 0.f;
    for (int i = 0; i < n; ++i) s += x[i];
    mu = s / n;
    for (int i = 0; i < n; ++i) s2 += (x[i] - mu) * (x[i] - mu);
    rs = rsqrtf(s2 / n + eps);
}

// z = act(x W1 + c1) W2 + c2 for the query in xq, or x + LN(that) with the inner
// norm; hbuf (m) and ybuf (d) are scratch
__device__ void mlp_query(const MlpF32Params &p, const float *xq, const float *W1, const float *c1,
                          const float *W2, const float *c2, float *hbuf, float *ybuf, float *zrow)
{
    const int d = p.d, m = p.m, tid = threadIdx.x;
    for (int j = tid; j < m; j += blockDim.x) {
        float s = c1[j];
        for (int i = 0; i < d; ++i) s = fmaf(xq[i], W1[i * m + j], s);
        hbuf[j] = act_f32(p.act, s);
    }
    __syncthreads();
    if (!p.ln_gamma) {
        for (int j = tid; j < d; j += blockDim.x) {
            float s = c2[j];
            for (int i = 0; i < m; ++i) s = fmaf(hbuf[i], W2[i * d + j], s);
            zrow[j] = s;
        }
        return;
    }
    // z = x + LN(y): y into ybuf, then every thread reads the row's statistics
    for (int j = tid; j < d; j += blockDim.x) {
        float s = c2[j];
        for (int i = 0; i < m; ++i) s = fmaf(hbuf[i], W2[i * d + j], s);
        ybuf[j] = s;
    }
    __syncthreads();
    float mu, rs;
    row_stats_f32(ybuf, d, p.ln_eps, mu, rs);
    const float *gm = p.ln_gamma + (size_t)(blockIdx.x % p.H) * d, *bt = p.ln_beta + (size_t)(blockIdx.x % p.H) * d;
    for (int j = tid; j < d; j += blockDim.x) zrow[j] = xq[j] + fmaf(gm[j], (ybuf[j] - mu) * rs, bt[j]);
}

__global__ void __launch_bounds__(kThreads) ttt_mlp_f32_kernel(const MlpF32Params p)
{
    extern __shared__ float sm[];
    const int d = p.d, m = p.m, T = p.T, tid = threadIdx.x, nt = blockDim.x;
    float *W1 = sm, *c1 = W1 + d * m, *W2 = c1 + m, *c2 = W2 + m * d;
    float *W1s = c2 + d, *c1s = W1s + d * m, *W2s = c1s + m, *c2s = W2s + m * d;
    float *hh = c2s + d, *aa = hh + m, *gg = aa + m, *hq = gg + m;
    float *kk = hq + m, *vv = kk + d, *qq = vv + d, *ee = qq + d, *yh = ee + d;
    const int bh = blockIdx.x;
    const bool ln = p.ln_gamma != nullptr;
    const float *gm = ln ? p.ln_gamma + (size_t)(bh % p.H) * d : nullptr;
    const float *bt = ln ? p.ln_beta + (size_t)(bh % p.H) * d : nullptr;
    const size_t ps = p.per_batch ? (size_t)bh : (size_t)(bh % p.H);
    for (int i = tid; i < d * m; i += nt) {
        W1[i] = p.W1[ps * d * m + i];
        W2[i] = p.W2[ps * m * d + i];
    }
    for (int i = tid; i < m; i += nt) c1[i] = p.c1[ps * m + i];
    for (int i = tid; i < d; i += nt) c2[i] = p.c2[ps * d + i];
    const float *q = p.q + (size_t)bh * T * d, *k = p.k + (size_t)bh * T * d;
    const float *v = p.v + (size_t)bh * T * d;
    float *z = p.z + (size_t)bh * T * d;

    for (int n0 = 0; n0 < T; n0 += p.b) {
        const int n1 = min(n0 + p.b, T);
        __syncthreads();
        for (int i = tid; i < d * m; i += nt) {
            W1s[i] = W1[i];
            W2s[i] = W2[i];
        }
        for (int i = tid; i < m; i += nt) c1s[i] = c1[i];
        for (int i = tid; i < d; i += nt) c2s[i] = c2[i];
        for (int t = n0; t < n1; ++t) {
            __syncthreads();
            for (int i = tid; i < d; i += nt) {
                kk[i] = k[(size_t)t * d + i];
                vv[i] = v[(size_t)t * d + i];
                qq[i] = q[(size_t)t * d + i];
            }
            __syncthreads();
            for (int j = tid; j < m; j += nt) {  // forward at the block start
                float s = c1s[j];
                for (int i = 0; i < d; ++i) s = fmaf(kk[i], W1s[i * m + j], s);
                hh[j] = s;
                aa[j] = act_f32(p.act, s);
            }
            __syncthreads();
            for (int j = tid; j < d; j += nt) {
                float s = c2s[j];
                for (int i = 0; i < m; ++i) s = fmaf(aa[i], W2s[i * d + j], s);
                ee[j] = ln ? s : s - vv[j];
            }
            if (ln) {  // e := dL/dy through x + LN(y): dy = (g - mean g - yh mean(g yh)) / s, g = gamma e
                __syncthreads();
                float mu, rs;
                row_stats_f32(ee, d, p.ln_eps, mu, rs);
                __syncthreads();  // every thread has read y
                for (int j = tid; j < d; j += nt) {
                    yh[j] = (ee[j] - mu) * rs;
                    ee[j] = gm[j] * (kk[j] + fmaf(gm[j], yh[j], bt[j]) - vv[j]);
                }
                __syncthreads();
                float mg = 0.f, mgy = 0.f;
                for (int j = 0; j < d; ++j) {
                    mg += ee[j];
                    mgy += ee[j] * yh[j];
                }
                __syncthreads();  // every thread has read g
                for (int j = tid; j < d; j += nt) ee[j] = (ee[j] - mg / d - yh[j] * (mgy / d)) * rs;
            }
            __syncthreads();
            for (int i = tid; i < m; i += nt) {  // g = (e W2s^T) * act'(h)
                float s = 0.f;
                for (int j = 0; j < d; ++j) s = fmaf(ee[j], W2s[i * d + j], s);
                gg[i] = s * act_d_f32(p.act, hh[i]);
            }
            __syncthreads();
            const float et = p.eta ? p.eta[(size_t)bh * T + t] : p.eta_scalar;
            for (int i = tid; i < m * d; i += nt) W2[i] = fmaf(-et * aa[i / d], ee[i % d], W2[i]);
            for (int i = tid; i < d * m; i += nt) W1[i] = fmaf(-et * kk[i / m], gg[i % m], W1[i]);
            for (int i = tid; i < d; i += nt) c2[i] = fmaf(-et, ee[i], c2[i]);
            for (int i = tid; i < m; i += nt) c1[i] = fmaf(-et, gg[i], c1[i]);
            if (p.causal) {
                __syncthreads();
                mlp_query(p, qq, W1, c1, W2, c2, hq, yh, z + (size_t)t * d);
            }
        }
        if (!p.causal) {
            for (int t = n0; t < n1; ++t) {
                __syncthreads();
                for (int i = tid; i < d; i += nt) qq[i] = q[(size_t)t * d + i];
                __syncthreads();
                mlp_query(p, qq, W1, c1, W2, c2, hq, yh, z + (size_t)t * d);
            }
        }
    }
    __syncthreads();
    if (p.W1o) for (int i = tid; i < d * m; i += nt) p.W1o[(size_t)bh * d * m + i] = W1[i];
    if (p.W2o) for (int i = tid; i < m * d; i += nt) p.W2o[(size_t)bh * m * d + i] = W2[i];
    if (p.c1o) for (int i = tid; i < m; i += nt) p.c1o[(size_t)bh * m + i] = c1[i];
    if (p.c2o) for (int i = tid; i < d; i += nt) p.c2o[(size_t)bh * d + i] = c2[i];
}

}  // namespace

bool mlp_f32_fits(int d, int m) { return mlp_f32_floats(d, m) * sizeof(float) <= 200u * 1024u; }

int launch_mlp_f32(const MlpArgs &a)
{
    if (!mlp_f32_fits(a.d, a.m)) return -2;
    const size_t smem = mlp_f32_floats(a.d, a.m) * sizeof(float);
    if (cudaFuncSetAttribute(ttt_mlp_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return -4;
    MlpF32Params p;
    p.H = a.H;
    p.T = a.T;
    p.d = a.d;
    p.m = a.m;
    p.b = a.b;
    p.causal = a.causal;
    p.per_batch = a.per_batch;
    p.act = a.act;
    p.ln_gamma = a.ln_gamma;
    p.ln_beta = a.ln_beta;
    p.ln_eps = a.ln_eps;
    p.q = static_cast<const float *>(a.q);
    p.k = static_cast<const float *>(a.k);
    p.v = static_cast<const float *>(a.v);
    p.eta = a.eta;
    p.eta_scalar = a.eta_scalar;
    p.W1 = a.W1;
    p.c1 = a.c1;
    p.W2 = a.W2;
    p.c2 = a.c2;
    p.z = static_cast<float *>(a.z);
    p.W1o = a.W1o;
    p.c1o = a.c1o;
    p.W2o = a.W2o;
    p.c2o = a.c2o;
    ttt_mlp_f32_kernel<<<a.B * a.H, kThreads, smem, a.stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace ttt
