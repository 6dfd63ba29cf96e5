// ttt_internal.h -- host-side launch interface between the C ABI (ttt_api.cu)
// and the kernels.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace ttt {

struct LinearArgs {
    int B, H, T, d, b, causal;
    const void *q, *k, *v;
    const float *eta;
    float eta_scalar;
    const float *W0;
    long long w0_bstride;
    void *z;
    float *W_out;
    int *status;         // device status word (timeouts)
    cudaStream_t stream;
};

struct MlpArgs {
    int B, H, T, d, m, b, causal, per_batch;
    const void *q, *k, *v;
    const float *eta;
    float eta_scalar;
    const float *W1, *c1, *W2, *c2;
    void *z;
    float *W1o, *c1o, *W2o, *c2o;
    int *status;
    cudaStream_t stream;
};

// Each returns 0 or a negative ttt_status code; maps = q, k, v tensor maps.
int launch_linear_bf16(const LinearArgs &a, const CUtensorMap *maps);
int launch_linear_f32(const LinearArgs &a);
int launch_mlp_f32(const MlpArgs &a);
int launch_mlp_bf16(const MlpArgs &a, const CUtensorMap *maps);
// Largest d*m the fp32 MLP path holds on chip.
bool mlp_f32_fits(int d, int m);

}  // namespace ttt
