// ttt_internal.h -- host-side launch interface between the C ABI (ttt_api.cu)
// and the kernels.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace ttt {

struct LinearArgs {
    int B, H, T, d, b, causal;
    int loss = 0, epochs = 1;  // loss: 0 MSE, 1 negative dot product; inner GD steps per mini-batch
    const float *ln_gamma = nullptr, *ln_beta = nullptr;  // inner norm [H][d] (null: f(x) = x W)
    float ln_eps = 1e-6f;
    const void *q, *k, *v;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    void *z;
    float *W_out;
    int *status;         // device status word (timeouts)
    cudaStream_t stream;
    // test hook (ttt_debug_wait_limit): > 0 makes the first consumer wait of the b = 16
    // and full-batch kernels wait this long on a barrier nothing arrives at
    unsigned long long test_stall_ns = 0;
};

struct MlpArgs {
    int B, H, T, d, m, b, causal, per_batch;
    int act = 0;  // inner activation: 0 SiLU, 1 GELU
    const float *ln_gamma = nullptr, *ln_beta = nullptr;  // inner norm [H][d] (null: plain MLP)
    float ln_eps = 1e-6f;
    const void *q, *k, *v;
    const float *eta;
    float eta_scalar;
    const float *W1, *c1, *W2, *c2;
    void *z;
    float *W1o, *c1o, *W2o, *c2o;
    int *status;
    cudaStream_t stream;
    unsigned long long test_stall_ns = 0;  // > 0: the timeout test (full-batch kernel)
};

struct DwconvArgs {
    int B, H, hh, ww, d, loss, epochs, bf16;
    const void *q, *k, *v;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    void *z;
    float *W_out;
    int *status;  // device status word (timeouts)
    cudaStream_t stream;
};

struct GateArgs {
    int B, T, H, dm;
    const void *x, *theta;  // bf16 [B][T][dm], [H][dm]
    float eta_base;
    float *eta;             // fp32 [B][H][T]
    int *status;            // device status word (timeouts)
    cudaStream_t stream;
};

// TMA descriptor of a bf16 token tensor viewed as [BH][T][d]: boxes of `rows`
// tokens x `cols` features (0: min(d, 64)), swizzled to the box row length, rows
// past T zero-filled on loads and dropped on stores.  Returns false if the driver
// entry point is unavailable or rejects it.
bool encode_token_map(CUtensorMap *m, const void *ptr, int BH, int T, int d, int rows, int cols = 0);

// Descriptor of a token tensor [BH][hh][ww][d] (bf16 or fp32) whose box is one
// sequence's zero-bordered grid: d x (ww+2) x (hh+2) at coordinates (0, -1, -1, bh),
// the border read as zeros (out of range).  False if d > 256, hh + 2 or ww + 2 > 256,
// or the encoding fails.
bool encode_grid_map(CUtensorMap *m, const void *ptr, bool bf16, int BH, int hh, int ww, int d);

// q, k, v descriptors (zeroed, unused when T == 0); false on an encoding failure.
inline bool encode_qkv(CUtensorMap *maps, const void *q, const void *k, const void *v, int BH, int T,
                       int d, int rows)
{
    for (int i = 0; i < 3; ++i)
        for (size_t j = 0; j < sizeof(CUtensorMap); ++j) reinterpret_cast<char *>(&maps[i])[j] = 0;
    if (T == 0) return true;
    return encode_token_map(&maps[0], q, BH, T, d, rows) && encode_token_map(&maps[1], k, BH, T, d, rows) &&
           encode_token_map(&maps[2], v, BH, T, d, rows);
}

// Each returns 0 or a negative ttt_status code.
int launch_linear_bf16(const LinearArgs &a);
int launch_linear_b16(const LinearArgs &a);  // b = 16 specialisation (d <= 64)
int launch_linear_b1(const LinearArgs &a);   // b = 1 (delta rule), column-parallel
int launch_linear_fb_tc(const LinearArgs &a);  // full batch, one epoch, on tcgen05
// b = 16, d <= 64 kernel over segments of each chain (segment 0 = tokens [0, len0),
// segment s >= 1 = [len0 + (s-1) seg_len, len0 + s seg_len)).  prep = false: output
// units for segments seg0 .. seg0+nseg-1 of every chain, from start weights W0
// (segment 0) or Wst (segment s: Wst[bh][s-1]).  prep = true: the state chain of
// segment 0 (its end weights to Wst[bh][0]) and the affine maps of segments
// 1 .. nsplit-2 (to mapbuf).  maps: the q, k, v descriptors (64-token boxes).
int launch_linear_b16_segments(const LinearArgs &a, int nsplit, int len0, int seg_len, int seg0, int nseg,
                               bool prep, float *Wst, float *mapbuf, const CUtensorMap *maps);
int launch_linear_fb(const LinearArgs &a);   // one full-batch mini-batch (b = T <= 256, non-causal, d = 64); -2 otherwise
int launch_linear_f32(const LinearArgs &a);
int launch_mlp_f32(const MlpArgs &a);
int launch_mlp_bf16(const MlpArgs &a);
// one full-batch mini-batch (b >= T, non-causal), d = 64, m = 256, on tcgen05; -2 otherwise
int launch_mlp_fb_tc(const MlpArgs &a);
// Sequence-parallel TTT-Linear (ttt_linear_seqpar.cu): the segment plan for a
// problem (false: the problem is not split, run the one-unit-per-chain path).
struct SeqparPlan {
    int nsplit = 0, len0 = 0, seg_len = 0;   // segments per chain, segment lengths
    size_t map_bytes = 0, wst_bytes = 0;     // scratch: affine maps, start weights
};
bool seqpar_plan(const LinearArgs &a, SeqparPlan &pl);
size_t seqpar_workspace_bytes(const SeqparPlan &pl);
// Enqueues the split forward on a.stream (forks a side stream and joins it back);
// ws: at least seqpar_workspace_bytes(pl) bytes of device memory, 256-byte aligned.
int launch_linear_seqpar(const LinearArgs &a, const SeqparPlan &pl, void *ws);
// The same split enqueued on a.stream alone: the preparing launch, the scan, then
// every segment's outputs in one launch (equal segments; seqpar_plan_serial).
bool seqpar_plan_serial(const LinearArgs &a, SeqparPlan &pl);
int launch_linear_seqpar_serial(const LinearArgs &a, const SeqparPlan &pl, void *ws);

// Depthwise 3x3 convolution inner model (ttt_dwconv.cu): shared memory bytes of
// one CTA and the launch.
size_t dwconv_smem(int hh, int ww, int d, int es);
int launch_dwconv(const DwconvArgs &a);
int launch_eta_gate(const GateArgs &a);  // H <= 64; -2 otherwise

// Largest d*m the fp32 MLP path holds on chip.
bool mlp_f32_fits(int d, int m);

}  // namespace ttt
