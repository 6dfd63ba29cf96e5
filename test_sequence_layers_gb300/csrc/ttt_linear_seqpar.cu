// ttt_linear_seqpar.cu -- sequence-parallel TTT-Linear forward (mini-batch b = 16,
// bf16 operands, fp32 state, d in {16, 32, 64}) for workloads with fewer
// (batch, head) chains than SMs, where one CTA per chain leaves most of the GPU
// idle and the serial mini-batch chain of a long sequence sets the time.
//
// One mini-batch step is affine in the weights:
//     W' = W - K^T diag(eta) (K W - V) = (I - K^T diag(eta) K) W + K^T diag(eta) V
// ("Learning to (Learn at Test Time)" walkthrough, section 1.2.2, mini-batch
// gradient descent, formula 6, written out for the linear inner model of section
// 2.2.1).  A run of steps is therefore one affine map W -> A W + B, and maps
// compose, so a chain can be cut into segments whose maps are found in parallel
// and chained by a short scan (the block-parallel remark of "Fast weights 与 TTT
// layers", on mini-batch versus exact sequential updates, made exact here: the
// maps reproduce the sequential mini-batch rule, not an approximation of it).
//
// Schedule, for nsplit segments per chain (segment 0 longer than the others):
//   caller's stream : outputs of segment 0 from W0 (ttt_linear_b16_kernel)
//   side stream     : the state chain of segment 0 alone (no query side: its end
//                     weights are segment 1's start) and, in the same launch, the
//                     affine maps of segments 1 .. nsplit-2
//                     -> scan: start weights of segments 2 .. nsplit-1 (fp32)
//                     -> outputs of segments 1 .. nsplit-1 from their start weights
// The side stream forks from and joins back into the caller's stream with events.
// Segment 0's output pass runs beside the side stream's first launch, so the
// segment lengths balance segment 0's output pass against that launch plus one
// output pass of a later segment.
//
// Scratch (caller-provided workspace): maps [BH][nsplit-2][2][d][d] fp32, then
// start weights [BH][nsplit-1][d][d] fp32.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ttt_device.cuh"
#include "ttt_internal.h"

namespace ttt {
namespace {

// Start weights of segments 2 .. nsplit-1 of one chain: W_{s+1} = A_s W_s + B_s
// in fp32, from W_1 (written by the state chain of segment 0).  One CTA of 256
// threads per chain, a 16 x 16 grid of threads each holding a TS x TS tile of the
// product (register blocking: per four steps along k, one 16-byte load of each of its
// rows of A and TS-wide loads of four rows of W feed 16 TS^2 FMAs).  The steps are
// serial, so the next map is fetched during the current product: A_{s+1} into the
// other shared buffer (cp.async), this thread's tile of B_{s+1} into registers.
template <int D>
__global__ void __launch_bounds__(256) ttt_linear_scan_kernel(const float *__restrict__ maps,
                                                              float *__restrict__ Wst, int nsplit)
{
    constexpr int TS = D / 16;  // tile side
    __shared__ __align__(16) float sW[D * D], sA[2][D * D];
    const int bh = blockIdx.x, t = threadIdx.x, ty = t / 16, tx = t % 16;
    const int r0 = TS * ty, c0 = TS * tx;
    float *W = Wst + (size_t)bh * (nsplit - 1) * D * D;
    auto map_a = [&](int s) { return maps + ((size_t)bh * (nsplit - 2) + s - 1) * 2 * D * D; };
    auto fetch_a = [&](int s, float *dst) {  // 16-byte pieces of A_s, committed as one group
        const float *A = map_a(s);
        for (int i = t; i < D * D / 4; i += 256) {
            const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst + 4 * i));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(A + 4 * i) : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    float bn[TS][TS];  // this thread's tile of the next B
    auto fetch_b = [&](int s) {
        const float *B = map_a(s) + D * D;
#pragma unroll
        for (int i = 0; i < TS; ++i)
#pragma unroll
            for (int j = 0; j < TS; ++j) bn[i][j] = B[(size_t)(r0 + i) * D + c0 + j];
    };
    for (int i = t; i < D * D; i += 256) sW[i] = W[i];
    if (nsplit > 2) {
        fetch_a(1, sA[0]);
        fetch_b(1);
    }
    for (int s = 1; s + 1 < nsplit; ++s) {
        const float *sa = sA[(s - 1) & 1];
        float acc[TS][TS];
#pragma unroll
        for (int i = 0; i < TS; ++i)
#pragma unroll
            for (int j = 0; j < TS; ++j) acc[i][j] = bn[i][j];
        if (s + 2 < nsplit) {  // the next map while this one multiplies
            fetch_a(s + 1, sA[s & 1]);
            fetch_b(s + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();  // A_s and the previous step's W are complete
#pragma unroll 4
        for (int k = 0; k < D; k += 4) {
            float4 a[TS];
#pragma unroll
            for (int i = 0; i < TS; ++i) a[i] = *reinterpret_cast<const float4 *>(sa + (r0 + i) * D + k);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float w[TS];
#pragma unroll
                for (int j = 0; j < TS; ++j) w[j] = sW[(k + kk) * D + c0 + j];
#pragma unroll
                for (int i = 0; i < TS; ++i) {
                    const float ak = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                    for (int j = 0; j < TS; ++j) acc[i][j] = fmaf(ak, w[j], acc[i][j]);
                }
            }
        }
        __syncthreads();  // every read of sW and of this step's A is done
        float *out = W + (size_t)s * D * D;
#pragma unroll
        for (int i = 0; i < TS; ++i)
#pragma unroll
            for (int j = 0; j < TS; ++j) {
                sW[(r0 + i) * D + c0 + j] = acc[i][j];
                out[(size_t)(r0 + i) * D + c0 + j] = acc[i][j];
            }
    }
}

int launch_scan(const LinearArgs &a, int nsplit, const float *maps, float *Wst, cudaStream_t st)
{
    const int BH = a.B * a.H;
    switch (a.d) {
    case 16: ttt_linear_scan_kernel<16><<<BH, 256, 0, st>>>(maps, Wst, nsplit); break;
    case 32: ttt_linear_scan_kernel<32><<<BH, 256, 0, st>>>(maps, Wst, nsplit); break;
    case 64: ttt_linear_scan_kernel<64><<<BH, 256, 0, st>>>(maps, Wst, nsplit); break;
    default: return -2;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Per device: the side stream and the fork / join events (created on first use).
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

std::mutex g_side_mu;
SideStream g_side[64];

// Per-chunk times of the two preparing roles relative to the output role (b = 16,
// d = 64, one CTA per SM), used to balance segment lengths: the state chain alone and
// a map (the chain on twice the columns).  The chain's ratio is fitted on the GB300 with
// the B2 H32 T32768 workload: 0.45 / 0.50 / 0.55 / 0.60 / 0.65 / 0.70 / 0.75 / 0.80 gave
// 336 / 334 / 329 / 325 / 336 / 349 / 362 / 376 us per call.
constexpr double kChainToOutput = 0.60;
constexpr double kMapToOutput = 0.95;

// The split's cost model, in units of one output-role chunk: the preparing roles' chunk
// costs, a fixed cost per launch and the scan's cost per map.  Mini-batches of 16: the
// ratios above (the fixed costs are small against the long sequences that split).
// Mini-batches of one token (the delta rule, whose chunks carry a forward substitution:
// 0.62 us per output chunk on the GB300): from the launch lists of linear_125m_b1, the
// state chain 0.86 and a map 1.85 of an output chunk (a map's eight warps share the
// sub-partitions) and about 5 us per launch.  The scan's 2.5 chunks per map is below the
// ~4 us a map took in those launch lists (6.5 chunks); for linear_125m_b1 both values
// give the same plan, while 6.5 would leave short two-chain sequences unsplit.
struct SplitCosts {
    double chain, map, launch, scan_map;
};
constexpr SplitCosts kCosts16 = {kChainToOutput, kMapToOutput, 0.0, 0.0};
constexpr SplitCosts kCosts1 = {0.86, 1.85, 8.0, 2.5};

// Modelled time (in output-chunk units) of a split with segment 0 of len0 tokens and
// nsplit - 1 later segments of len1 tokens: segment 0's outputs on the caller's stream
// against the preparing launch, the scan (with maps) and the later segments' outputs on
// the side stream.
double split_time(int len0, int len1, int nsplit, const SplitCosts &k)
{
    const double c0 = len0 / 16.0, c1 = len1 / 16.0;
    double prep = c0 * k.chain;
    if (nsplit > 2 && c1 * k.map > prep) prep = c1 * k.map;
    const double scan = nsplit > 2 ? k.launch + (nsplit - 2) * k.scan_map : 0.0;
    const double later = k.launch + prep + scan + k.launch + c1;
    const double first = k.launch + c0;
    return first > later ? first : later;
}

}  // namespace

bool seqpar_plan(const LinearArgs &a, SeqparPlan &pl)
{
    pl = SeqparPlan{};
    // (the inner norm makes a step non-affine in W: no maps).  Mini-batches of 16, or of
    // one token (the delta rule, in 16-token chunks: each chunk is affine in W as well)
    if ((a.b != 16 && a.b != 1) || (a.d != 16 && a.d != 32 && a.d != 64) || a.loss != 0 || a.epochs != 1 ||
        a.ln_gamma)
        return false;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    const long long BH = (long long)a.B * a.H;
    const int T = a.T;
    // segment 0's output CTAs and the side stream's first launch (BH chain CTAs and
    // BH (nsplit - 2) map CTAs) share the GPU: nsplit BH <= SMs
    int pmax = (int)(nsm / (BH > 0 ? BH : 1));
    if (pmax > 8) pmax = 8;
    const SplitCosts &kc = a.b == 1 ? kCosts1 : kCosts16;
    double best = (kc.launch + T / 16.0) * 0.9;  // a split must save at least a tenth
    for (int P = 2; P <= pmax; ++P) {
        for (int len0 = 64; len0 < T; len0 += 64) {
            const int rest = T - len0;
            const int len1 = ((rest + (P - 1) - 1) / (P - 1) + 63) / 64 * 64;
            if (len1 < (a.b == 1 ? 128 : 256)) continue;  // segments too short to pay
            const int nseg = 1 + (rest + len1 - 1) / len1;
            const double t = split_time(len0, len1, nseg, kc);
            if (t < best) {
                best = t;
                pl.nsplit = nseg;
                pl.len0 = len0;
                pl.seg_len = len1;
            }
        }
    }
    if (pl.nsplit < 2) return false;
    const size_t dd = (size_t)a.d * a.d * sizeof(float);
    pl.map_bytes = (size_t)BH * (pl.nsplit - 2) * 2 * dd;
    pl.wst_bytes = (size_t)BH * (pl.nsplit - 1) * dd;
    return true;
}

size_t seqpar_workspace_bytes(const SeqparPlan &pl)
{
    return pl.nsplit < 2 ? 0 : ((pl.map_bytes + 255) / 256) * 256 + pl.wst_bytes;
}

int launch_linear_seqpar(const LinearArgs &a, const SeqparPlan &pl, void *ws)
{
    float *maps = static_cast<float *>(ws);
    float *Wst = reinterpret_cast<float *>(static_cast<char *>(ws) + ((pl.map_bytes + 255) / 256) * 256);
    CUtensorMap tm[3];
    if (!encode_qkv(tm, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 64)) return -4;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -4;
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream &S = g_side[dev];
    if (!S.s) {
        if (cudaStreamCreateWithFlags(&S.s, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&S.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&S.join, cudaEventDisableTiming) != cudaSuccess)
            return -4;
    }
    if (cudaEventRecord(S.fork, a.stream) != cudaSuccess || cudaStreamWaitEvent(S.s, S.fork, 0) != cudaSuccess)
        return -4;
    // caller's stream: segment 0 from W0
    int rc = launch_linear_b16_segments(a, pl.nsplit, pl.len0, pl.seg_len, 0, 1, false, Wst, maps, tm);
    // side stream: segment 0's state chain (+ maps of segments 1 .. nsplit-2) -> scan -> segments 1 ..
    LinearArgs b = a;
    b.stream = S.s;
    if (rc == 0) rc = launch_linear_b16_segments(b, pl.nsplit, pl.len0, pl.seg_len, 0, 1, true, Wst, maps, tm);
    if (rc == 0 && pl.nsplit > 2) rc = launch_scan(b, pl.nsplit, maps, Wst, S.s);
    if (rc == 0)
        rc = launch_linear_b16_segments(b, pl.nsplit, pl.len0, pl.seg_len, 1, pl.nsplit - 1, false, Wst, maps, tm);
    // join (also after a failed launch, so the caller's stream never runs ahead of
    // work already queued on the side stream)
    if (cudaEventRecord(S.join, S.s) != cudaSuccess || cudaStreamWaitEvent(a.stream, S.join, 0) != cudaSuccess)
        return -4;
    return rc;
}

// Plan for a split run on one stream (no side stream): the preparing launch first,
// then the scan, then the outputs of all segments in one launch.  Segments of
// equal length; time = preparing pass + one segment's output pass.
bool seqpar_plan_serial(const LinearArgs &a, SeqparPlan &pl)
{
    pl = SeqparPlan{};
    if ((a.b != 16 && a.b != 1) || (a.d != 16 && a.d != 32 && a.d != 64) || a.loss != 0 || a.epochs != 1 ||
        a.ln_gamma)
        return false;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    const long long BH = (long long)a.B * a.H;
    const int T = a.T;
    int pmax = (int)(nsm / (BH > 0 ? BH : 1));  // the output launch: nsplit BH CTAs
    if (pmax > 8) pmax = 8;
    double best = T / 16.0 * 0.9;  // a split must save at least a tenth
    for (int P = 2; P <= pmax; ++P) {
        const int len = ((T + P - 1) / P + 63) / 64 * 64;
        if (len < 256) break;
        const int nseg = (T + len - 1) / len;
        if (nseg < 2) continue;
        const double c = len / 16.0;
        const double t = c * (nseg > 2 ? kMapToOutput : kChainToOutput) + c;
        if (t < best) {
            best = t;
            pl.nsplit = nseg;
            pl.len0 = pl.seg_len = len;
        }
    }
    if (pl.nsplit < 2) return false;
    const size_t dd = (size_t)a.d * a.d * sizeof(float);
    pl.map_bytes = (size_t)BH * (pl.nsplit - 2) * 2 * dd;
    pl.wst_bytes = (size_t)BH * (pl.nsplit - 1) * dd;
    return true;
}

int launch_linear_seqpar_serial(const LinearArgs &a, const SeqparPlan &pl, void *ws)
{
    float *maps = static_cast<float *>(ws);
    float *Wst = reinterpret_cast<float *>(static_cast<char *>(ws) + ((pl.map_bytes + 255) / 256) * 256);
    CUtensorMap tm[3];
    if (!encode_qkv(tm, a.q, a.k, a.v, a.B * a.H, a.T, a.d, 64)) return -4;
    int rc = launch_linear_b16_segments(a, pl.nsplit, pl.len0, pl.seg_len, 0, 1, true, Wst, maps, tm);
    if (rc == 0 && pl.nsplit > 2) rc = launch_scan(a, pl.nsplit, maps, Wst, a.stream);
    if (rc == 0)
        rc = launch_linear_b16_segments(a, pl.nsplit, pl.len0, pl.seg_len, 0, pl.nsplit, false, Wst, maps, tm);
    return rc;
}

}  // namespace ttt
