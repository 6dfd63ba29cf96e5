/*
 * ttt.h -- C ABI of libttt: forward pass (prefill / inference) of a
 * Test-Time-Training (TTT) layer on one NVIDIA GB300 (sm_103a).
 *
 * The layer.  For every (batch, head) sequence the hidden state is the weight set W
 * of a small inner model f(x; W).  W starts at W0 and is trained on the sequence
 * itself by gradient descent on the reconstruction loss
 *     l_t(W) = 1/2 || f(k_t; W) - v_t ||^2
 * ("Fast weights 与 TTT layers", opening formula; "TTT：Test-Time Training",
 * section TTT, MSE loss).  Tokens are taken in consecutive mini-batches of b
 * tokens; every token of a mini-batch takes its gradient at the W that the previous
 * mini-batch left ("Learning to (Learn at Test Time)" walkthrough, section 1.2.2,
 * mini-batch gradient descent, formula 6).  The output is z_t = f(q_t; W_t)
 * (same walkthrough, section 1.2, output rule), where
 *   causal = 1:  W_t = W_start - sum_{s in t's mini-batch, s <= t} eta_s grad l_s(W_start)
 *                (the cumulative-sum channel of section 1.2.2: W_t includes token
 *                t's own write);
 *   causal = 0:  every query of a mini-batch reads the W at the end of that
 *                mini-batch (b = T gives one full-batch step, the vision variant of
 *                the ViT3 article, observation 2).
 * b = 1 is the delta rule ("Fast weights 与 TTT layers", section 1).
 *
 * Inner models (walkthrough section 2.2.1; ViT3 article, observations 4 and 6):
 *   ttt_linear_fwd:  f(x; W) = x W,                      W in R^{d x d}
 *   ttt_mlp_fwd:     f(x) = act(x W1 + c1) W2 + c2,       W1 d x m, W2 m x d
 *   ttt_dwconv_fwd:  a depthwise 3 x 3 convolution over a token grid
 *   (optionally x + LN(f(x)) for the first two: the inner norm and residual).
 * ttt_eta_gate computes the per-token rates eta = eta_base * sigma(theta_lr . x)
 * from the layer input (walkthrough section 2.2.3) in the layout the others read.
 * Row convention throughout: a token x is a 1 x d row vector.
 *
 * Conventions shared by every entry point
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory.  Its device state is one small status word per
 *     device and the fixed 4 MiB scratch array of ttt_linear_fwd_seqpar_noalloc
 *     (a static device array, held on every device that loads the library until
 *     the process exits).
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream) and runs asynchronously.  The return value reports
 *     argument validation and launch errors synchronously.  A kernel-side wait that
 *     timed out (never expected; every on-chip wait is bounded to about 2 s) is
 *     reported by ttt_sync_status().
 *   - Layouts are C-contiguous: q, k, v, z are [B, H, T, d] in io_dtype; eta is
 *     [B, H, T] fp32; weights are fp32.
 *   - Alignment: q, k, v, z must be 16-byte aligned (TTT_ERR_ALIGN otherwise);
 *     eta and the fp32 weight arrays 4-byte aligned.
 *   - T may be 0 (then only the final weights are written, equal to the initial
 *     ones) and need not be a multiple of b: the last mini-batch is shorter.
 *   - Final-weight outputs may be NULL (not written).  They may alias the
 *     corresponding initial-weight inputs when those are given per (batch, head)
 *     (in-place continuation of a sequence); they may not overlap shared
 *     ([H, ...]) initial weights (TTT_ERR_ARG).
 */
#ifndef TTT_H_
#define TTT_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TTT_OK = 0,
    TTT_ERR_ARG = -1,          /* null / negative / inconsistent argument            */
    TTT_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. d not in the set)   */
    TTT_ERR_ALIGN = -3,        /* pointer misaligned for the bulk-copy engine         */
    TTT_ERR_LAUNCH = -4,       /* CUDA reported an error at or before launch          */
    TTT_ERR_TIMEOUT = -5,      /* a kernel wait ran out (reported by ttt_sync_status) */
    TTT_ERR_SCRATCH = -6       /* ttt_linear_fwd_seqpar_noalloc: more than its fixed scratch */
} ttt_status;

typedef enum { TTT_F32 = 0, TTT_BF16 = 1 } ttt_dtype;

/* Inner loss of TTT-Linear.
 *   TTT_LOSS_MSE: l_t(W) = 1/2 || k_t W - v_t ||^2 (the reconstruction loss above).
 *   TTT_LOSS_DOT: l_t(W) = -(k_t W) . v_t, the negative dot product ("TTT：Test-Time
 *                 Training", section 如何理解; the inner loss of the ViT3 block).  Its
 *                 gradient -k_t^T v_t does not depend on W, so the layer becomes
 *                 linear attention with state W0 + sum eta_s k_s^T v_s. */
typedef enum { TTT_LOSS_MSE = 0, TTT_LOSS_DOT = 1 } ttt_loss;

/* TTT-Linear problem description. */
typedef struct {
    int B, H, T, d;            /* batch, heads, tokens, head dim (d in {16,32,64,128}) */
    int mini_batch;            /* b >= 1                                               */
    int causal;                /* 1 causal, 0 non-causal (queries read block-end W)    */
    ttt_dtype io_dtype;        /* dtype of q, k, v and z                               */
    long long w0_batch_stride; /* elements between batches of W0; 0 = W0 is [H,d,d]
                                  shared by every batch entry, H*d*d = [B,H,d,d]       */
    int loss;                  /* ttt_loss (0 = TTT_LOSS_MSE)                          */
    int epochs;                /* inner gradient steps on the mini-batch: 0 or 1 = one;
                                  > 1 (the ViT3 article's inner epochs) needs causal = 0
                                  and mini_batch >= T, every query reading the last W;
                                  bf16 supports it for d = 64, T <= 256
                                  (TTT_ERR_UNSUPPORTED otherwise)                       */
    const float *ln_gamma;     /* inner layer norm + residual: f(x) = x + LN(x W) with
                                  LN(y) = ln_gamma * (y - mean) / sqrt(var + ln_eps)
                                  + ln_beta over the d outputs ("Learning to (Learn at
                                  Test Time)" walkthrough, section 2.2.1); [H,d] fp32
                                  device arrays, fixed (not trained by the inner step),
                                  or both NULL for f(x) = x W.  MSE loss and one epoch
                                  only; bf16 needs mini_batch 16 and d <= 64
                                  (TTT_ERR_UNSUPPORTED otherwise)                       */
    const float *ln_beta;
    float ln_eps;              /* > 0 when the norm is used (1e-6 in the paper's code)  */
} ttt_linear_desc;

/*
 * TTT-Linear forward.
 *   q, k, v : [B,H,T,d] io_dtype (queries, keys = training view, values = labels)
 *   eta     : [B,H,T] fp32 per-token learning rate of the writing token, or NULL to
 *             use eta_scalar for every token (walkthrough section 2.2.3)
 *   W0      : fp32 initial weights, W0[i][j] multiplies input i into output j
 *   z       : [B,H,T,d] io_dtype output
 *   W_out   : [B,H,d,d] fp32 final weights, or NULL
 * io_dtype TTT_BF16 runs the tensor-core path: bf16 operands, fp32 accumulation and
 * fp32 weight state.  TTT_F32 runs an fp32 CUDA-core path (no reduced precision).
 */
ttt_status ttt_linear_fwd(const ttt_linear_desc *desc,
                          const void *q, const void *k, const void *v,
                          const float *eta, float eta_scalar,
                          const float *W0, void *z, float *W_out, void *stream);

/*
 * Sequence-parallel TTT-Linear forward: the same results as ttt_linear_fwd (up to the
 * order of floating-point rounding), for problems with fewer (batch, head) chains
 * than the GPU has SMs and long sequences.
 *
 * One mini-batch step is affine in the weights, W' = (I - K^T diag(eta) K) W +
 * K^T diag(eta) V ("Learning to (Learn at Test Time)" walkthrough, section 1.2.2,
 * formula 6, for the linear inner model of section 2.2.1), so each chain is cut
 * into segments of whole 64-token blocks: the affine maps W -> A W + B of the
 * segments are computed in parallel, a scan turns them into every segment's start
 * weights, and the segments' outputs are computed in parallel from those.  The
 * first segment runs from W0 while the maps are formed.
 *
 * Applies to io_dtype TTT_BF16 with mini_batch 16, or 1 (the delta rule, whose
 * 16-token chunks are affine in the weights as well), d in {16, 32, 64} and the MSE
 * loss, when the GPU has at least two SMs per chain; otherwise the call runs
 * ttt_linear_fwd (workspace unused, may be NULL).
 *   workspace       : device scratch owned by the caller, 256-byte aligned, at least
 *                     ttt_linear_seqpar_workspace(desc) bytes; it holds the maps and
 *                     start weights and must not be touched until the work queued
 *                     on `stream` has finished.
 * The work is queued on `stream`; internally it forks to a second stream of the
 * library's own (one per device, created on the first split call) and joins back
 * with events, so later work on `stream` sees the outputs.  W_out must not overlap
 * W0 here (TTT_ERR_ARG): the first segment may still read W0 while the last one
 * writes W_out.  TTT_ERR_ARG also for a missing, misaligned or too small workspace.
 */
size_t ttt_linear_seqpar_workspace(const ttt_linear_desc *desc);

ttt_status ttt_linear_fwd_seqpar(const ttt_linear_desc *desc,
                                 const void *q, const void *k, const void *v,
                                 const float *eta, float eta_scalar,
                                 const float *W0, void *z, float *W_out,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * ttt_linear_fwd_seqpar_noalloc: the sequence-parallel forward without a caller
 * workspace and without any device allocation.  (The pages have no counterpart:
 * this is a deployment variant of ttt_linear_fwd_seqpar.)
 *
 * For callers that cannot allocate device memory while they run: a serving
 * process that has handed the free device memory to its own pool or cache has none
 * left for cudaMalloc, cudaFree may synchronise the device in the middle of its
 * pipeline, and a plugin inside another framework may have no access to that
 * framework's allocator.  The scratch is instead a fixed array of 4 MiB inside the
 * library, held on every device that loads it until the process exits.
 *
 * Same arguments and results as ttt_linear_fwd_seqpar (up to floating-point
 * rounding), all work on `stream` alone: one launch for the first segment's state
 * chain and the later segments' affine maps, the scan, then every segment's
 * outputs in one launch (segments of equal length).  Problems that do not split
 * run ttt_linear_fwd.  A split needs 4 (BH (P-1) + 2 BH (P-2)) d^2 bytes for P
 * segments of BH = B*H chains (e.g. d = 64, two segments: up to 256 chains);
 * larger problems return TTT_ERR_SCRATCH before any work is queued.  W_out must
 * not overlap W0 (TTT_ERR_ARG).
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call uses the same array: calls whose work overlaps on the GPU
 * (other streams, other host threads) race on it and must be ordered by the
 * caller.  Nothing in the array needs clearing between calls.
 */
ttt_status ttt_linear_fwd_seqpar_noalloc(const ttt_linear_desc *desc,
                                         const void *q, const void *k, const void *v,
                                         const float *eta, float eta_scalar,
                                         const float *W0, void *z, float *W_out, void *stream);

/* Inner activation of TTT-MLP.
 *   TTT_ACT_SILU: SiLU(h) = h sigma(h) (the ViT3 article, observation 4).
 *   TTT_ACT_GELU: GELU(h) = h Phi(h), Phi the standard normal CDF, in its exact
 *                 (erf) form (the walkthrough's TTT-MLP, section 2.2.1). */
typedef enum { TTT_ACT_SILU = 0, TTT_ACT_GELU = 1 } ttt_activation;

/* TTT-MLP problem description. */
typedef struct {
    int B, H, T, d, m;         /* d in {16,32,64}; m = hidden width, multiple of 16    */
    int mini_batch;            /* b >= 1                                               */
    int causal;
    ttt_dtype io_dtype;
    int params_per_batch;      /* 0: W1,c1,W2,c2 are [H,...] shared over the batch;
                                  1: they are [B,H,...]                                */
    int activation;            /* ttt_activation (0 = TTT_ACT_SILU)                    */
    const float *ln_gamma;     /* inner layer norm + residual: f(x) = x + LN(act(x W1 +
                                  c1) W2 + c2), LN over the d outputs as in
                                  ttt_linear_desc ("Learning to (Learn at Test Time)"
                                  walkthrough, section 2.2.1); [H,d] fp32 device arrays,
                                  fixed, or both NULL for the plain MLP.  bf16 I/O needs
                                  d = 64, m = 256 and mini_batch <= 16 or one
                                  non-causal full batch (mini_batch >= T); otherwise
                                  TTT_ERR_UNSUPPORTED                                   */
    const float *ln_beta;
    float ln_eps;              /* > 0 when the norm is used                             */
} ttt_mlp_desc;

/*
 * TTT-MLP forward, f(x) = act(x W1 + c1) W2 + c2, act = SiLU or GELU (desc->activation),
 * or x + LN(f(x)) with the inner norm (desc->ln_gamma, ln_beta, ln_eps).
 *   W1 [..,d,m], c1 [..,m], W2 [..,m,d], c2 [..,d] fp32 initial inner weights;
 *   the *_out arrays are [B,H,...] fp32 final weights (each may be NULL).
 * Other arguments as for ttt_linear_fwd.
 */
ttt_status ttt_mlp_fwd(const ttt_mlp_desc *desc,
                       const void *q, const void *k, const void *v,
                       const float *eta, float eta_scalar,
                       const float *W1, const float *c1, const float *W2, const float *c2,
                       void *z, float *W1_out, float *c1_out, float *W2_out, float *c2_out,
                       void *stream);

/* Depthwise-convolution TTT problem description. */
typedef struct {
    int B, H;                  /* batch, heads                                          */
    int height, width;         /* token grid: N = height * width tokens per sequence,
                                  row-major (token y * width + x)                       */
    int d;                     /* channels per head, a multiple of 8                    */
    ttt_dtype io_dtype;        /* dtype of q, k, v and z                                */
    int loss;                  /* ttt_loss                                              */
    int epochs;                /* full-batch inner steps, >= 1                          */
    long long w0_batch_stride; /* 0: W0 is [H,9,d] shared over the batch; H*9*d: [B,H,9,d] */
} ttt_dwconv_desc;

/*
 * TTT with a depthwise 3x3 convolution as the inner model, full-batch inner GD over
 * all N tokens, non-causal (the ViT3 article, observation 6, a small convolution as
 * the inner model of vision TTT, and observation 2, full-batch inner training):
 *     f(X; W)[p][c] = sum_{o = (di+1)*3 + (dj+1), di, dj in {-1,0,1}} X[p + (di,dj)][c] W[o][c]
 * on the token grid with zero padding.  Each epoch takes the gradient of
 * sum_p eta_p l_p at the epoch's start taps and steps by it; z = f(q; W_final).
 *   q, k, v, z : [B,H,N,d] io_dtype; eta: [B,H,N] fp32 or NULL (eta_scalar)
 *   W0         : fp32 taps, see w0_batch_stride; W_out: [B,H,9,d] fp32 or NULL
 * The sequence is held on chip: two padded grids of (height+2) (width+2) d
 * sizeof(io) bytes and V of N d sizeof(io) bytes, each rounded up to 128 bytes, plus
 * 256 + 4 (9 d + N + 9 * 512) bytes must fit in 227 KB (bf16, d = 64: up to 22 x 22
 * tokens), else TTT_ERR_UNSUPPORTED.  Pointers: q, k,
 * v, z 16-byte aligned (TTT_ERR_ALIGN), fp32 arrays 4-byte aligned.
 */
ttt_status ttt_dwconv_fwd(const ttt_dwconv_desc *desc,
                          const void *q, const void *k, const void *v,
                          const float *eta, float eta_scalar,
                          const float *W0, void *z, float *W_out, void *stream);

/* Input-dependent inner learning rate problem description. */
typedef struct {
    int B, T;                  /* batch, tokens per sequence                            */
    int H;                     /* heads, 1 .. 64 (TTT_ERR_UNSUPPORTED above)            */
    int dm;                    /* width of the layer's input tokens, a multiple of 8
                                  (TTT_ERR_UNSUPPORTED otherwise)                       */
} ttt_gate_desc;

/*
 * The inner learning rate as a function of the input token ("Learning to (Learn at
 * Test Time)" walkthrough, section 2.2.3): a learnable vector of the outer loop per
 * head, a sigmoid, and a base rate (1 for TTT-Linear, 0.1 for TTT-MLP):
 *     eta[b,h,t] = eta_base * sigma(theta[h] . x[b,t]),  sigma(a) = 1 / (1 + e^-a)
 *   x     : [B,T,dm] bf16, the layer's input tokens, 16-byte aligned
 *   theta : [H,dm] bf16, one vector per head, 16-byte aligned
 *   eta   : [B,H,T] fp32 (written), 4-byte aligned: the per-token rates that
 *           ttt_linear_fwd, ttt_linear_fwd_seqpar and ttt_mlp_fwd read
 * The dot products accumulate in fp32 from the bf16 operands.  All pointers are
 * device memory owned by the caller; eta must not overlap x or theta (TTT_ERR_ARG).
 * B = 0 or T = 0 queues nothing.  Misaligned pointers: TTT_ERR_ALIGN.
 */
ttt_status ttt_eta_gate(const ttt_gate_desc *desc, const void *x, const void *theta, float eta_base,
                        float *eta, void *stream);

/* Waits for `stream`, then reports (and clears) a kernel wait timeout recorded on
 * the current device, or a CUDA error seen while waiting. */
ttt_status ttt_sync_status(void *stream);

/* Static description of a status code. */
const char *ttt_status_str(ttt_status s);

/* Number of kernel launches this library has enqueued on the calling process
 * (all devices); used to count this library's launches inside a timed region. */
unsigned long long ttt_launch_count(void);

/*
 * Test hook of the timeout path (never needed in normal use; the pages have no
 * counterpart).  With ns > 0, every later TTT-Linear launch of the b = 16 kernel
 * (causal or not, mini_batch 16, d <= 64) and of the full-batch kernel (bf16, d = 64,
 * mini_batch >= T <= 256, one epoch) makes its first consumer-side wait on a barrier
 * that nothing arrives at, bounded by ns nanoseconds: the wait runs out, the kernel
 * records TTT_ERR_TIMEOUT in the device status word, skips its products (outputs
 * undefined), still waits for its own copies in flight and frees its tensor memory,
 * and ttt_sync_status() reports the timeout.  ns = 0 restores normal operation.  The
 * setting is process-wide (read at each launch); other kernels ignore it.
 */
void ttt_debug_wait_limit(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* TTT_H_ */
