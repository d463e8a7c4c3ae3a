// Router GEMV + hard gate (SwiAttn report, section 2, router design):
// logit_t = <h_t, w> + b, gate_t = 1(sigmoid(logit_t) > 0.5) = 1(logit_t > 0).
// HBM-bound: each warp takes two tokens at a time (route_gemv.cuh).

#include "route_gemv.cuh"
#include "swiattn_internal.h"

#include <cuda_bf16.h>

namespace swi {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) route_kernel(const uint4* __restrict__ h,
                                                    const uint4* __restrict__ w, float bias,
                                                    int64_t tokens, int nvec,
                                                    float* __restrict__ logits,
                                                    uint8_t* __restrict__ gate) {
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    int64_t t = warp0;
    for (; t + nwarps < tokens; t += 2 * nwarps) route_token2<T>(h, w, bias, t, t + nwarps, nvec, logits, gate);
    if (t < tokens) route_token<T>(h, w, bias, t, nvec, logits, gate);
}

}  // namespace

cudaError_t launch_route(const void* h, const void* w, float bias, int64_t tokens, int d_model,
                         int dtype, float* logits, uint8_t* gate, cudaStream_t s) {
    if (tokens == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (tokens + 7) / 8;   // 8 warps per block, one token per warp
    const int blocks = static_cast<int>(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    if (dtype == 1) {
        route_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            static_cast<const uint4*>(h), static_cast<const uint4*>(w), bias, tokens, d_model / 8,
            logits, gate);
    } else {
        route_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(h),
                                                   static_cast<const uint4*>(w), bias, tokens,
                                                   d_model / 4, logits, gate);
    }
    return cudaGetLastError();
}

}  // namespace swi
