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
// CUDA cores.  A persistent CTA walks the sequences (batch, head) with K, Q and V
// of one sequence in shared memory in the I/O type; with two buffers the next
// sequence's copies are in flight while the current one computes.  K and Q sit in
// zero-bordered grids, so the taps need no bounds tests; one TMA copy per grid
// writes the border as out-of-range zeros (larger d: one bulk copy per grid row
// and a border zeroed once).  Each thread owns a pair of channels and an even run
// of positions, walks it with a 3 x 3 register window (three new taps per
// position instead of nine), forms each residual on the fly and accumulates the
// nine tap gradients with the paired fp32 FMA; the per-thread partial sums are
// reduced through shared memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "ttt_device.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

struct DwParams {
    int BH, H, hh, ww, d, dot, epochs, tma;  // tma: grid boxes through the tensor maps
    const void *q, *k, *v;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    void *z;
    float *W_out;
    int *status;
};

// Threads of a CTA holding NB sequence buffers (one CTA per SM when NB == 2, two
// when NB == 1).
template <int NB>
constexpr int dw_threads = 256 * NB;

__host__ __device__ inline size_t round128(size_t x) { return (x + 127) & ~(size_t)127; }

// Shared memory of a CTA with nb sequence buffers, from a 128-byte aligned base:
// 128 bytes of mbarriers ([nb][2]: K and V, Q); per buffer the K grid, the Q grid
// (each (hh+2) x (ww+2) x d, I/O type) and V [N][d], each padded to 128 bytes; then
// taps W [nb][9][d], partial tap gradients [parts][9][d] (paired 8-byte accesses,
// so ahead of the odd-length eta) and eta [nb][N].
struct DwLayout {
    size_t grid, vbytes, buf, total;  // total includes 128 bytes of alignment slack
    int parts;
};

__host__ __device__ inline DwLayout dw_layout(int hh, int ww, int d, int es, int nb)
{
    DwLayout L;
    L.grid = round128((size_t)(hh + 2) * (ww + 2) * d * es);
    L.vbytes = round128((size_t)hh * ww * d * es);
    L.buf = 2 * L.grid + L.vbytes;
    L.parts = 256 * nb / (d / 2);
    L.total = 256 + nb * L.buf + 4 * (nb * 9 * (size_t)d + (size_t)L.parts * 9 * d + (size_t)nb * hh * ww);
    return L;
}

template <typename TIO>
__device__ __forceinline__ float2 ld2(const TIO *p)
{
    if constexpr (sizeof(TIO) == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
        return make_float2(bf16_lo(w), bf16_hi(w));
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

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes a multiple of
// 16), completion counted on the mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// TMA: 4-D tiled tensor load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, uint32_t bar, int c0, int c1, int c2,
                                            int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int PENDING>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
}

// zero border (rows 0 and hh+1, columns 0 and ww+1) of a padded grid, in 16-byte
// pieces (a cell is d * sizeof(TIO) bytes, a multiple of 16)
template <typename TIO>
__device__ __forceinline__ void zero_border(TIO *grid, int hh, int ww, int d)
{
    const int gw = ww + 2, vpc = d * (int)sizeof(TIO) / 16;
    uint4 *g4 = reinterpret_cast<uint4 *>(grid);
    for (int i = threadIdx.x; i < 2 * (gw + hh) * vpc; i += blockDim.x) {
        const int cell = i / vpc, piece = i - cell * vpc;
        int y, x;
        if (cell < gw) { y = 0; x = cell; }
        else if (cell < 2 * gw) { y = hh + 1; x = cell - gw; }
        else { const int r = cell - 2 * gw; y = 1 + (r >> 1); x = (r & 1) ? ww + 1 : 0; }
        g4[(y * gw + x) * vpc + piece] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Walks the positions p0 .. p1-1 (row-major) of a padded grid with a 3 x 3 window
// for channel pair c, one row segment at a time.  The window's columns rotate
// through three register triples (unrolled by three, so no moves);
// step(pos, a, b, n) gets the padded columns x, x+1, x+2 of padded rows y .. y+2
// for output (y, x) = pos, i.e. tap (r, j) is {a, b, n}[j][r].  Offsets within a
// sequence fit in 32 bits; with d a compile-time constant the column offsets
// become immediates.
template <typename TIO, typename Step>
__device__ __forceinline__ void walk_run(const TIO *g, int p0, int p1, int ww, int d, int c, Step &&step)
{
    const int gw = ww + 2;
    int y = p0 < p1 ? p0 / ww : 0, x0 = p0 - y * ww;  // (ww > 0 whenever the run is not empty)
    while (p0 < p1) {
        const int x1 = min(ww, x0 + (p1 - p0)), base = y * ww;
        const TIO *r0 = g + y * gw * d + c, *r1 = r0 + gw * d, *r2 = r1 + gw * d;
        float2 A[3], B[3], C[3];
        auto col = [&](int xc, float2 (&cc)[3]) {
            cc[0] = ld2(r0 + xc * d);
            cc[1] = ld2(r1 + xc * d);
            cc[2] = ld2(r2 + xc * d);
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
        const float2 vv = ld2(sV + pos * d + c);
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

// Issues (warp 0) the copies of sequence bh's tokens into one buffer; K and V
// complete on kv, Q on qb.  TMA path: one box per grid (the border arrives as
// out-of-range zeros) and one bulk copy for V, from lane 0.  Otherwise one bulk
// copy per grid row (the interior of a padded row is contiguous) and one for V.
// The buffer was last read through the generic proxy, hence the proxy fence.
template <typename TIO>
__device__ __forceinline__ void issue_tokens(const DwParams &p, const CUtensorMap *tmk, const CUtensorMap *tmq, int bh,
                                             TIO *sK, TIO *sQ, TIO *sV, uint32_t kv, uint32_t qb)
{
    const int lane = threadIdx.x, hh = p.hh, ww = p.ww, d = p.d, gw = ww + 2;
    const uint32_t row = (uint32_t)(ww * d * sizeof(TIO)), vbytes = (uint32_t)hh * row;
    const size_t off = (size_t)bh * hh * ww * d;
    fence_proxy_async();
    if (p.tma) {
        if (lane == 0) {
            const uint32_t box = (uint32_t)((hh + 2) * gw * d * sizeof(TIO));
            mbar_arrive_expect_tx(kv, box + vbytes);
            mbar_arrive_expect_tx(qb, box);
            tma_load_4d(smem_u32(sK), tmk, kv, 0, -1, -1, bh);
            tma_load_4d(smem_u32(sQ), tmq, qb, 0, -1, -1, bh);
            bulk_load(smem_u32(sV), static_cast<const TIO *>(p.v) + off, vbytes, kv);
        }
        return;
    }
    if (lane == 0) {
        mbar_arrive_expect_tx(kv, 2u * vbytes);
        mbar_arrive_expect_tx(qb, vbytes);
    }
    __syncwarp();
    if (hh > 0 && ww > 0) {
        const TIO *gk = static_cast<const TIO *>(p.k) + off, *gq = static_cast<const TIO *>(p.q) + off;
        for (int y = lane; y < hh; y += 32) {
            const uint32_t o = (uint32_t)(((y + 1) * gw + 1) * d * sizeof(TIO));
            bulk_load(smem_u32(sK) + o, gk + (size_t)y * ww * d, row, kv);
            bulk_load(smem_u32(sQ) + o, gq + (size_t)y * ww * d, row, qb);
        }
        if (lane == 0) bulk_load(smem_u32(sV), static_cast<const TIO *>(p.v) + off, vbytes, kv);
    }
}

// Asynchronous 4-byte copies (every thread) of sequence bh's start taps and
// per-token eta; the caller commits them as one group.
__device__ __forceinline__ void issue_small(const DwParams &p, int bh, int d, float *sW, float *sEta)
{
    const int N = p.hh * p.ww;
    const float *W0 = p.W0 + (size_t)(bh / p.H) * p.w0_bstride + (size_t)(bh % p.H) * 9 * d;
    for (int i = threadIdx.x; i < 9 * d; i += blockDim.x) cp_async_4(smem_u32(sW + i), W0 + i);
    if (p.eta)
        for (int i = threadIdx.x; i < N; i += blockDim.x) cp_async_4(smem_u32(sEta + i), p.eta + (size_t)bh * N + i);
}

// CTAs walk the sequences blockIdx.x, blockIdx.x + gridDim.x, ...  With two
// buffers the next sequence's copies are in flight while the current one
// computes.  DC > 0 fixes d at compile time.
template <typename TIO, int NB, int DC>
__global__ void __launch_bounds__(dw_threads<NB>, 3 - NB) ttt_dwconv_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq, const DwParams p)
{
    constexpr int NT = dw_threads<NB>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    // 128-byte aligned base for the TMA destinations (the size includes the slack)
    unsigned char *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const int d = DC > 0 ? DC : p.d, hh = p.hh, ww = p.ww, N = hh * ww;
    const DwLayout L = dw_layout(hh, ww, d, (int)sizeof(TIO), NB);
    const int gbytes = (int)L.grid, bbytes = (int)L.buf;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // [NB][2]: K and V, Q
    unsigned char *buf = smem + 128;
    float *sW0 = reinterpret_cast<float *>(buf + NB * bbytes);  // 128-byte aligned
    float *sPart = sW0 + NB * 9 * d;                           // 8-byte aligned (d % 8 == 0)
    const int npair = d / 2, parts = NT / npair;
    float *sEta0 = sPart + parts * 9 * d;
    const int tid = threadIdx.x, part = tid / npair, c = 2 * (tid % npair);
    auto gK = [&](int b) { return reinterpret_cast<TIO *>(buf + b * bbytes); };
    auto gQ = [&](int b) { return reinterpret_cast<TIO *>(buf + b * bbytes + gbytes); };
    auto gV = [&](int b) { return reinterpret_cast<TIO *>(buf + b * bbytes + 2 * gbytes); };
    auto bkv = [&](int b) { return smem_u32(bars + 2 * b); };
    auto bq = [&](int b) { return smem_u32(bars + 2 * b + 1); };

    if (tid == 0) {
        for (int b = 0; b < NB; ++b) {
            mbar_init(bkv(b), 1);
            mbar_init(bq(b), 1);
        }
        fence_barrier_init();
    }
    if (!p.tma)  // row copies write only the grid interiors; the border stays zero
        for (int b = 0; b < NB; ++b) {
            zero_border(gK(b), hh, ww, d);
            zero_border(gQ(b), hh, ww, d);
        }
    __syncthreads();

    const bool active = tid < parts * npair;
    // this thread's run of positions: an even share of the N in row-major order
    const int p0 = (int)((long long)N * part / parts), p1 = (int)((long long)N * (part + 1) / parts);
    // W -= upd * (summed partials): the dot loss's sign and a scalar eta
    const float upd = (p.dot ? -1.f : 1.f) * (p.eta ? 1.f : p.eta_scalar);

    int bh = blockIdx.x, last = -1;  // last: local index of the newest sequence issued
    auto issue = [&](int jj, int seq) {
        const int b = jj % NB;
        if (tid < 32) issue_tokens<TIO>(p, &tmk, &tmq, seq, gK(b), gQ(b), gV(b), bkv(b), bq(b));
        issue_small(p, seq, d, sW0 + b * 9 * d, sEta0 + b * N);
        last = jj;
    };
    // after a timeout (never expected): wait, bounded, for every copy still in flight
    auto drain = [&]() {
        for (int jj = last - NB + 1 < 0 ? 0 : last - NB + 1; jj <= last; ++jj) {
            mbar_wait(bkv(jj % NB), (jj / NB) & 1, p.status, kSiteStage);
            mbar_wait(bq(jj % NB), (jj / NB) & 1, p.status, kSiteStage);
        }
        cp_async_wait<0>();
    };
    if (bh < p.BH) issue(0, bh);
    cp_async_commit();

    for (int j = 0; bh < p.BH; bh += gridDim.x, ++j) {
        const int b = j % NB;
        const uint32_t par = (j / NB) & 1;
        float *sW = sW0 + b * 9 * d, *sEta = sEta0 + b * N;
        // NB == 2: the next sequence's copies go out now, into the buffer the previous
        // sequence released at its final barrier; NB == 1: the current sequence's
        // (after the first), once that barrier has passed
        const int nj = NB == 2 ? j + 1 : j, nbh = NB == 2 ? bh + (int)gridDim.x : bh;
        if (nj > last && nbh < p.BH) issue(nj, nbh);
        cp_async_commit();
        if constexpr (NB == 2) cp_async_wait<1>();  // this thread's taps and eta of sequence j
        else cp_async_wait<0>();
        // K and V landed (every thread observes the barrier), every thread's small
        // copies are visible; a timeout is CTA-uniform after the vote
        if (!__syncthreads_and(mbar_wait(bkv(b), par, p.status, kSiteStage))) {
            drain();
            return;
        }
        const TIO *sK = gK(b), *sV = gV(b);
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
                for (int o = 0; o < 9; ++o) *reinterpret_cast<float2 *>(sPart + (part * 9 + o) * d + c) = g[o];
            }
            __syncthreads();  // partial sums visible; every read of sW is done
            for (int i = tid; i < 9 * d; i += NT) {
                float s = 0.f;
                for (int r = 0; r < parts; ++r) s += sPart[r * 9 * d + i];
                sW[i] = fmaf(-upd, s, sW[i]);
            }
            __syncthreads();  // the epoch's taps visible
        }

        // output pass over the Q grid
        if (!__syncthreads_and(mbar_wait(bq(b), par, p.status, kSiteStage))) {
            drain();
            return;
        }
        if (active) {
            float2 w[9];
#pragma unroll
            for (int o = 0; o < 9; ++o) w[o] = *reinterpret_cast<const float2 *>(sW + o * d + c);
            TIO *z = static_cast<TIO *>(p.z) + (size_t)bh * N * d;
            walk_run(gQ(b), p0, p1, ww, d, c,
                     [&](int pos, const float2(&a)[3], const float2(&bb)[3], const float2(&n)[3]) {
                         float2 zz = make_float2(0.f, 0.f);
#pragma unroll
                         for (int r = 0; r < 3; ++r) {
                             zz = fma2(a[r], w[3 * r], zz);
                             zz = fma2(bb[r], w[3 * r + 1], zz);
                             zz = fma2(n[r], w[3 * r + 2], zz);
                         }
                         st2(z + pos * d + c, zz.x, zz.y);
                     });
        }
        if (p.W_out)
            for (int i = tid; i < 9 * d; i += NT) p.W_out[(size_t)bh * 9 * d + i] = sW[i];
        __syncthreads();  // buffer b, its taps and eta, and the partials released
    }
}

// Persistent launch: as many CTAs as fit on the device at once, at most one per
// sequence.
template <typename TIO, int NB, int DC>
int launch_nb(const CUtensorMap &tmk, const CUtensorMap &tmq, const DwParams &p, size_t smem, cudaStream_t st)
{
    auto kern = ttt_dwconv_kernel<TIO, NB, DC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return -4;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, dw_threads<NB>, smem) != cudaSuccess || per_sm < 1)
        return -4;
    const long long slots = (long long)sms * per_sm;
    const int grid = (int)(p.BH < slots ? p.BH : slots);
    kern<<<grid, dw_threads<NB>, smem, st>>>(tmk, tmq, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// d = 64 (the ViT3-style head dimension) with compile-time strides
template <typename TIO, int NB>
int launch_d(const CUtensorMap &tmk, const CUtensorMap &tmq, const DwParams &p, size_t smem, cudaStream_t st)
{
    return p.d == 64 ? launch_nb<TIO, NB, 64>(tmk, tmq, p, smem, st) : launch_nb<TIO, NB, 0>(tmk, tmq, p, smem, st);
}

}  // namespace

// The API's size limit is the single-buffer layout's.
size_t dwconv_smem(int hh, int ww, int d, int es) { return dw_layout(hh, ww, d, es, 1).total; }

int launch_dwconv(const DwconvArgs &a)
{
    DwParams p;
    CUtensorMap tmk, tmq;  // zero-bordered grid boxes of K and Q (used when p.tma != 0)
    std::memset(&p, 0, sizeof p);
    std::memset(&tmk, 0, sizeof tmk);
    std::memset(&tmq, 0, sizeof tmq);
    p.BH = a.B * a.H;
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
    // one TMA box per grid where the descriptors allow it (d <= 256), else row copies
    p.tma = a.hh > 0 && a.ww > 0 && encode_grid_map(&tmk, a.k, a.bf16, p.BH, a.hh, a.ww, a.d) &&
            encode_grid_map(&tmq, a.q, a.bf16, p.BH, a.hh, a.ww, a.d);
    // two buffers (prefetch of the next sequence) whenever they fit in 227 KB
    const int es = a.bf16 ? 2 : 4;
    const size_t smem2 = dw_layout(a.hh, a.ww, a.d, es, 2).total, smem1 = dw_layout(a.hh, a.ww, a.d, es, 1).total;
    const bool two = smem2 <= 227 * 1024;
    if (a.bf16)
        return two ? launch_d<__nv_bfloat16, 2>(tmk, tmq, p, smem2, a.stream)
                   : launch_d<__nv_bfloat16, 1>(tmk, tmq, p, smem1, a.stream);
    return two ? launch_d<float, 2>(tmk, tmq, p, smem2, a.stream) : launch_d<float, 1>(tmk, tmq, p, smem1, a.stream);
}

}  // namespace ttt
