// ttt_api.cu -- the C ABI declared in include/ttt.h: argument validation, TMA
// descriptor encoding, kernel dispatch and the per-device status word.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ttt.h"
#include "ttt_internal.h"

// Status word written by kernels whose bounded on-chip wait ran out (one per
// device: every device that loads the library has its own copy).
__device__ int g_ttt_status;

// Fixed scratch of ttt_linear_fwd_seqpar_noalloc (affine maps and segment start
// weights of a split run).  Every device that loads the library holds it until the
// process exits.  Every byte a call reads from it is written earlier by the same
// call, so it never needs clearing.
constexpr size_t kNoAllocScratchBytes = 4u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::atomic<unsigned long long> g_launches{0};
std::atomic<unsigned long long> g_test_stall_ns{0};  // ttt_debug_wait_limit

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Address of this device's status word (looked up once per device).
int *status_word()
{
    static std::mutex mu;
    static int *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ttt_status) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<int *>(p);
    }
    return addr[dev];
}

// Device address of this device's fixed scratch array.  The array's name in host
// code only stands for the symbol: the address comes from cudaGetSymbolAddress,
// looked up once per device with that device current (nullptr on failure).
void *noalloc_scratch()
{
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

// q/k/v viewed as a 3-D tensor [B*H][T][d] of bf16; box = `rows` tokens x min(d,64)
// features, swizzled to the box row length so that ldmatrix is conflict-free.
bool ttt::encode_token_map(CUtensorMap *m, const void *ptr, int BH, int T, int d, int rows, int cols)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    if (cols <= 0) cols = d < 64 ? d : 64;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
    const cuuint32_t box[3] = {(cuuint32_t)cols, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    // swizzle span = the box row length (128, 64 or 32 bytes)
    const CUtensorMapSwizzle sw = cols >= 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool ttt::encode_grid_map(CUtensorMap *m, const void *ptr, bool bf16, int BH, int hh, int ww, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || d > 256 || ww + 2 > 256 || hh + 2 > 256) return false;
    const cuuint64_t es = bf16 ? 2 : 4;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)ww, (cuuint64_t)hh, (cuuint64_t)BH};
    const cuuint64_t strides[3] = {(cuuint64_t)d * es, (cuuint64_t)ww * d * es, (cuuint64_t)hh * ww * d * es};
    const cuuint32_t box[4] = {(cuuint32_t)d, (cuuint32_t)ww + 2, (cuuint32_t)hh + 2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(ptr),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

ttt_status code(int rc) { return static_cast<ttt_status>(rc); }

}  // namespace

namespace {

// Validates a TTT-Linear call and fills the launch arguments (status TTT_OK or the
// error to return).
ttt_status linear_args(const ttt_linear_desc *desc, const void *q, const void *k, const void *v,
                       const float *eta, float eta_scalar, const float *W0, void *z, float *W_out,
                       void *stream, ttt::LinearArgs &a)
{
    if (!desc) return TTT_ERR_ARG;
    const ttt_linear_desc D = *desc;
    if (D.B < 1 || D.H < 1 || D.T < 0 || D.mini_batch < 1 || !W0) return TTT_ERR_ARG;
    if (D.causal != 0 && D.causal != 1) return TTT_ERR_ARG;
    if (D.io_dtype != TTT_F32 && D.io_dtype != TTT_BF16) return TTT_ERR_ARG;
    if (D.T > 0 && (!q || !k || !v || !z)) return TTT_ERR_ARG;
    if (D.d != 16 && D.d != 32 && D.d != 64 && D.d != 128) return TTT_ERR_UNSUPPORTED;
    if (D.loss != TTT_LOSS_MSE && D.loss != TTT_LOSS_DOT) return TTT_ERR_ARG;
    if (D.epochs < 0) return TTT_ERR_ARG;
    if (D.epochs > 1 && (D.causal || D.mini_batch < D.T)) return TTT_ERR_UNSUPPORTED;
    const bool ln = D.ln_gamma || D.ln_beta;
    if (ln && (!D.ln_gamma || !D.ln_beta || !(D.ln_eps > 0.f) || D.loss != TTT_LOSS_MSE)) return TTT_ERR_ARG;
    if (ln && (!aligned(D.ln_gamma, 4) || !aligned(D.ln_beta, 4))) return TTT_ERR_ALIGN;
    if (ln && D.epochs > 1) return TTT_ERR_UNSUPPORTED;
    const long long dd = (long long)D.d * D.d;
    if (D.w0_batch_stride != 0 && D.w0_batch_stride != (long long)D.H * dd) return TTT_ERR_ARG;
    if ((long long)D.B * D.H > 0x7fffffffLL) return TTT_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16)) return TTT_ERR_ALIGN;
    if (!aligned(W0, 4) || !aligned(eta, 4) || !aligned(W_out, 4)) return TTT_ERR_ALIGN;
    if (W_out && D.w0_batch_stride == 0 &&
        overlaps(W_out, sizeof(float) * dd * D.B * D.H, W0, sizeof(float) * dd * D.H))
        return TTT_ERR_ARG;

    a.B = D.B;
    a.H = D.H;
    a.T = D.T;
    a.d = D.d;
    a.b = D.T > 0 && D.mini_batch > D.T ? D.T : D.mini_batch;  // b >= T is one block
    a.causal = D.causal;
    a.loss = D.loss;
    a.epochs = D.epochs > 1 ? D.epochs : 1;
    a.ln_gamma = ln ? D.ln_gamma : nullptr;
    a.ln_beta = ln ? D.ln_beta : nullptr;
    a.ln_eps = D.ln_eps;
    a.q = q;
    a.k = k;
    a.v = v;
    a.eta = eta;
    a.eta_scalar = eta_scalar;
    a.W0 = W0;
    a.w0_bstride = D.w0_batch_stride;
    a.z = z;
    a.W_out = W_out;
    a.status = status_word();
    a.stream = static_cast<cudaStream_t>(stream);
    a.test_stall_ns = g_test_stall_ns.load(std::memory_order_relaxed);
    if (!a.status) return TTT_ERR_LAUNCH;
    return TTT_OK;
}

int launch_linear(const ttt::LinearArgs &a, ttt_dtype io)
{
    int rc;
    if (io == TTT_BF16 && a.ln_gamma) {  // inner norm: the b = 16 kernel only (one mini-batch of
                                         // T <= 16 tokens is one of its chunks)
        const bool b16 = a.b == 16 || (a.b == a.T && a.T < 16);
        rc = (b16 && a.d <= 64) ? ttt::launch_linear_b16(a) : TTT_ERR_UNSUPPORTED;
    } else if (io == TTT_BF16) {
        rc = ttt::launch_linear_fb_tc(a);  // full-batch mini-batch: no serial chain
        if (rc == TTT_ERR_UNSUPPORTED) rc = ttt::launch_linear_fb(a);  // several epochs
        if (rc == TTT_ERR_UNSUPPORTED && a.epochs == 1)  // repeated epochs: the full-batch kernel only
            rc = (a.b == 1 && a.d <= 64 && !a.loss) ? ttt::launch_linear_b16(a)  // delta rule in 16-token chunks
                 : a.b == 1                          ? ttt::launch_linear_b1(a)   // column-parallel
                 : (a.b == 16 && a.d <= 64)          ? ttt::launch_linear_b16(a)
                                                     : ttt::launch_linear_bf16(a);
    } else
        rc = ttt::launch_linear_f32(a);
    return rc;
}

// The split plan of a validated bf16 call (nsplit 0: not split).
ttt::SeqparPlan seqpar_plan_for(const ttt_linear_desc *desc, const ttt::LinearArgs &a)
{
    ttt::SeqparPlan pl;
    if (desc->io_dtype != TTT_BF16 || !ttt::seqpar_plan(a, pl)) pl = ttt::SeqparPlan{};
    return pl;
}

}  // namespace

extern "C" {

ttt_status ttt_linear_fwd(const ttt_linear_desc *desc, const void *q, const void *k, const void *v,
                          const float *eta, float eta_scalar, const float *W0, void *z,
                          float *W_out, void *stream)
{
    ttt::LinearArgs a;
    const ttt_status st = linear_args(desc, q, k, v, eta, eta_scalar, W0, z, W_out, stream, a);
    if (st != TTT_OK) return st;
    const int rc = launch_linear(a, desc->io_dtype);
    if (rc == 0) g_launches.fetch_add(1, std::memory_order_relaxed);
    return code(rc);
}

size_t ttt_linear_seqpar_workspace(const ttt_linear_desc *desc)
{
    if (!desc || desc->B < 1 || desc->H < 1 || desc->T < 1 || desc->mini_batch < 1) return 0;
    ttt::LinearArgs a{};
    a.B = desc->B;
    a.H = desc->H;
    a.T = desc->T;
    a.d = desc->d;
    a.b = desc->mini_batch > desc->T ? desc->T : desc->mini_batch;
    a.loss = desc->loss;
    a.epochs = desc->epochs > 1 ? desc->epochs : 1;
    a.ln_gamma = desc->ln_gamma;
    return ttt::seqpar_workspace_bytes(seqpar_plan_for(desc, a));
}

ttt_status ttt_linear_fwd_seqpar(const ttt_linear_desc *desc, const void *q, const void *k, const void *v,
                                 const float *eta, float eta_scalar, const float *W0, void *z,
                                 float *W_out, void *workspace, size_t workspace_bytes, void *stream)
{
    ttt::LinearArgs a;
    const ttt_status st = linear_args(desc, q, k, v, eta, eta_scalar, W0, z, W_out, stream, a);
    if (st != TTT_OK) return st;
    const ttt::SeqparPlan pl = seqpar_plan_for(desc, a);
    int rc, n = 1;
    if (pl.nsplit < 2) {
        rc = launch_linear(a, desc->io_dtype);
    } else {
        const size_t need = ttt::seqpar_workspace_bytes(pl);
        if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return TTT_ERR_ARG;
        // the first segment reads W0 while the last one writes W_out on another stream
        const size_t dd = sizeof(float) * desc->d * desc->d;
        const size_t nW0 = desc->w0_batch_stride ? dd * desc->B * desc->H : dd * desc->H;
        if (W_out && overlaps(W_out, dd * desc->B * desc->H, W0, nW0)) return TTT_ERR_ARG;
        if (overlaps(workspace, need, z, (size_t)desc->B * desc->H * desc->T * desc->d * 2)) return TTT_ERR_ARG;
        rc = ttt::launch_linear_seqpar(a, pl, workspace);
        n = pl.nsplit > 2 ? 4 : 3;  // segment 0, chain (+ maps), scan, later segments
    }
    if (rc == 0) g_launches.fetch_add(n, std::memory_order_relaxed);
    return code(rc);
}

ttt_status ttt_mlp_fwd(const ttt_mlp_desc *desc, const void *q, const void *k, const void *v,
                       const float *eta, float eta_scalar, const float *W1, const float *c1,
                       const float *W2, const float *c2, void *z, float *W1_out, float *c1_out,
                       float *W2_out, float *c2_out, void *stream)
{
    if (!desc) return TTT_ERR_ARG;
    const ttt_mlp_desc D = *desc;
    if (D.B < 1 || D.H < 1 || D.T < 0 || D.mini_batch < 1 || D.m < 1) return TTT_ERR_ARG;
    if (!W1 || !c1 || !W2 || !c2) return TTT_ERR_ARG;
    if (D.causal != 0 && D.causal != 1) return TTT_ERR_ARG;
    if (D.params_per_batch != 0 && D.params_per_batch != 1) return TTT_ERR_ARG;
    if (D.activation != TTT_ACT_SILU && D.activation != TTT_ACT_GELU) return TTT_ERR_ARG;
    if (D.io_dtype != TTT_F32 && D.io_dtype != TTT_BF16) return TTT_ERR_ARG;
    if (D.T > 0 && (!q || !k || !v || !z)) return TTT_ERR_ARG;
    const bool ln = D.ln_gamma || D.ln_beta;
    if (ln && (!D.ln_gamma || !D.ln_beta || !(D.ln_eps > 0.f))) return TTT_ERR_ARG;
    if (D.d != 16 && D.d != 32 && D.d != 64) return TTT_ERR_UNSUPPORTED;
    if (D.m % 16 != 0) return TTT_ERR_UNSUPPORTED;
    if (ln && D.io_dtype == TTT_BF16 &&  // the bf16 inner norm: d = 64, m = 256, mini-batches of at
        (D.d != 64 || D.m != 256 ||      // most 16 tokens or one non-causal full batch
         ((D.T > 0 && D.mini_batch > D.T ? D.T : D.mini_batch) > 16 && (D.causal || D.mini_batch < D.T))))
        return TTT_ERR_UNSUPPORTED;
    if (ln && (!aligned(D.ln_gamma, 4) || !aligned(D.ln_beta, 4))) return TTT_ERR_ALIGN;
    if ((long long)D.B * D.H > 0x7fffffffLL) return TTT_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16)) return TTT_ERR_ALIGN;
    const void *f32p[] = {eta, W1, c1, W2, c2, W1_out, c1_out, W2_out, c2_out};
    for (const void *p : f32p)
        if (!aligned(p, 4)) return TTT_ERR_ALIGN;
    if (!D.params_per_batch) {
        const size_t nH = (size_t)D.H, nBH = (size_t)D.B * D.H, dm = (size_t)D.d * D.m;
        const struct { const void *o; size_t no; const void *i; size_t ni; } pairs[] = {
            {W1_out, nBH * dm, W1, nH * dm}, {c1_out, nBH * D.m, c1, nH * D.m},
            {W2_out, nBH * dm, W2, nH * dm}, {c2_out, nBH * D.d, c2, nH * D.d}};
        for (const auto &pr : pairs)
            if (pr.o && overlaps(pr.o, 4 * pr.no, pr.i, 4 * pr.ni)) return TTT_ERR_ARG;
    }

    ttt::MlpArgs a;
    a.test_stall_ns = g_test_stall_ns.load(std::memory_order_relaxed);
    a.B = D.B;
    a.H = D.H;
    a.T = D.T;
    a.d = D.d;
    a.m = D.m;
    a.b = D.T > 0 && D.mini_batch > D.T ? D.T : D.mini_batch;
    a.causal = D.causal;
    a.per_batch = D.params_per_batch;
    a.act = D.activation;
    a.ln_gamma = ln ? D.ln_gamma : nullptr;
    a.ln_beta = ln ? D.ln_beta : nullptr;
    a.ln_eps = D.ln_eps;
    a.q = q;
    a.k = k;
    a.v = v;
    a.eta = eta;
    a.eta_scalar = eta_scalar;
    a.W1 = W1;
    a.c1 = c1;
    a.W2 = W2;
    a.c2 = c2;
    a.z = z;
    a.W1o = W1_out;
    a.c1o = c1_out;
    a.W2o = W2_out;
    a.c2o = c2_out;
    a.status = status_word();
    a.stream = static_cast<cudaStream_t>(stream);
    if (!a.status) return TTT_ERR_LAUNCH;

    int rc;
    if (D.io_dtype == TTT_BF16)
        rc = ttt::launch_mlp_bf16(a);
    else
        rc = ttt::launch_mlp_f32(a);
    if (rc == 0) g_launches.fetch_add(1, std::memory_order_relaxed);
    return code(rc);
}

ttt_status ttt_linear_fwd_seqpar_noalloc(const ttt_linear_desc *desc, const void *q, const void *k,
                                         const void *v, const float *eta, float eta_scalar, const float *W0,
                                         void *z, float *W_out, void *stream)
{
    ttt::LinearArgs a;
    const ttt_status st = linear_args(desc, q, k, v, eta, eta_scalar, W0, z, W_out, stream, a);
    if (st != TTT_OK) return st;
    ttt::SeqparPlan pl;
    if (desc->io_dtype != TTT_BF16 || !ttt::seqpar_plan_serial(a, pl)) {
        const int rc = launch_linear(a, desc->io_dtype);  // not split: needs no scratch
        if (rc == 0) g_launches.fetch_add(1, std::memory_order_relaxed);
        return code(rc);
    }
    if (ttt::seqpar_workspace_bytes(pl) > kNoAllocScratchBytes) return TTT_ERR_SCRATCH;
    const size_t dd = sizeof(float) * desc->d * desc->d;
    const size_t nW0 = desc->w0_batch_stride ? dd * desc->B * desc->H : dd * desc->H;
    if (W_out && overlaps(W_out, dd * desc->B * desc->H, W0, nW0)) return TTT_ERR_ARG;
    void *ws = noalloc_scratch();
    if (!ws) return TTT_ERR_LAUNCH;
    const int rc = ttt::launch_linear_seqpar_serial(a, pl, ws);
    if (rc == 0) g_launches.fetch_add(pl.nsplit > 2 ? 3 : 2, std::memory_order_relaxed);
    return code(rc);
}

ttt_status ttt_dwconv_fwd(const ttt_dwconv_desc *desc, const void *q, const void *k, const void *v,
                          const float *eta, float eta_scalar, const float *W0, void *z, float *W_out,
                          void *stream)
{
    if (!desc) return TTT_ERR_ARG;
    const ttt_dwconv_desc D = *desc;
    if (D.B < 1 || D.H < 1 || D.height < 0 || D.width < 0 || D.d < 1 || D.epochs < 1 || !W0)
        return TTT_ERR_ARG;
    if (D.io_dtype != TTT_F32 && D.io_dtype != TTT_BF16) return TTT_ERR_ARG;
    if (D.loss != TTT_LOSS_MSE && D.loss != TTT_LOSS_DOT) return TTT_ERR_ARG;
    const long long N = (long long)D.height * D.width;
    if (N > 0 && (!q || !k || !v || !z)) return TTT_ERR_ARG;
    if (D.w0_batch_stride != 0 && D.w0_batch_stride != (long long)D.H * 9 * D.d) return TTT_ERR_ARG;
    if (D.d % 8 != 0 || D.d > 512 || (long long)D.B * D.H > 0x7fffffffLL || N > (1 << 20))
        return TTT_ERR_UNSUPPORTED;
    if (ttt::dwconv_smem(D.height, D.width, D.d, D.io_dtype == TTT_BF16 ? 2 : 4) > 227 * 1024)
        return TTT_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16)) return TTT_ERR_ALIGN;
    if (!aligned(W0, 4) || !aligned(eta, 4) || !aligned(W_out, 4)) return TTT_ERR_ALIGN;
    ttt::DwconvArgs a;
    a.B = D.B;
    a.H = D.H;
    a.hh = D.height;
    a.ww = D.width;
    a.d = D.d;
    a.loss = D.loss;
    a.epochs = D.epochs;
    a.bf16 = D.io_dtype == TTT_BF16;
    a.q = q;
    a.k = k;
    a.v = v;
    a.eta = eta;
    a.eta_scalar = eta_scalar;
    a.W0 = W0;
    a.w0_bstride = D.w0_batch_stride;
    a.z = z;
    a.W_out = W_out;
    a.status = status_word();
    a.stream = static_cast<cudaStream_t>(stream);
    if (!a.status) return TTT_ERR_LAUNCH;
    const int rc = ttt::launch_dwconv(a);
    if (rc == 0) g_launches.fetch_add(1, std::memory_order_relaxed);
    return code(rc);
}

ttt_status ttt_eta_gate(const ttt_gate_desc *desc, const void *x, const void *theta, float eta_base,
                        float *eta, void *stream)
{
    if (!desc) return TTT_ERR_ARG;
    const ttt_gate_desc D = *desc;
    if (D.B < 0 || D.T < 0 || D.H < 1 || D.dm < 1) return TTT_ERR_ARG;
    if (D.B == 0 || D.T == 0) return TTT_OK;
    if (!x || !theta || !eta) return TTT_ERR_ARG;
    if (D.H > 64 || D.dm % 8 != 0 || D.B > 65535) return TTT_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(theta, 16) || !aligned(eta, 4)) return TTT_ERR_ALIGN;
    const size_t nx = (size_t)D.B * D.T * D.dm * 2, nth = (size_t)D.H * D.dm * 2, ne = (size_t)D.B * D.H * D.T * 4;
    if (overlaps(eta, ne, x, nx) || overlaps(eta, ne, theta, nth)) return TTT_ERR_ARG;
    ttt::GateArgs a;
    a.B = D.B;
    a.T = D.T;
    a.H = D.H;
    a.dm = D.dm;
    a.x = x;
    a.theta = theta;
    a.eta_base = eta_base;
    a.eta = eta;
    a.status = status_word();
    a.stream = static_cast<cudaStream_t>(stream);
    if (!a.status) return TTT_ERR_LAUNCH;
    const int rc = ttt::launch_eta_gate(a);
    if (rc == 0) g_launches.fetch_add(1, std::memory_order_relaxed);
    return code(rc);
}

ttt_status ttt_sync_status(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TTT_ERR_LAUNCH;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_ttt_status, sizeof(int)) != cudaSuccess) return TTT_ERR_LAUNCH;
    if (v != 0) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_ttt_status, &zero, sizeof(int));
        return TTT_ERR_TIMEOUT;
    }
    return TTT_OK;
}

const char *ttt_status_str(ttt_status s)
{
    switch (s) {
    case TTT_OK: return "ok";
    case TTT_ERR_ARG: return "invalid argument";
    case TTT_ERR_UNSUPPORTED: return "unsupported configuration";
    case TTT_ERR_ALIGN: return "pointer misaligned (q, k, v, z need 16 bytes; fp32 arrays 4)";
    case TTT_ERR_LAUNCH: return "CUDA error at launch";
    case TTT_ERR_TIMEOUT: return "kernel wait timed out";
    case TTT_ERR_SCRATCH: return "the split run needs more than the library's fixed 4 MiB scratch";
    }
    return "unknown status";
}

unsigned long long ttt_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void ttt_debug_wait_limit(unsigned long long ns) { g_test_stall_ns.store(ns, std::memory_order_relaxed); }

}  // extern "C"
