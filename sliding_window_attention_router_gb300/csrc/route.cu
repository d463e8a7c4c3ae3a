// Router GEMV + hard gate (SwiAttn report, section 2, router design):
// logit_t = <h_t, w> + b, gate_t = 1(sigmoid(logit_t) > 0.5) = 1(logit_t > 0).
// HBM-bound: one warp per token streams its hidden row with 16-byte loads.

#include "swiattn_internal.h"

#include <cuda_bf16.h>

namespace swi {
namespace {

__device__ __forceinline__ float dot16(const uint4& a, const uint4& b, __nv_bfloat16) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float2 u = __bfloat1622float2(x[t]);
        const float2 v = __bfloat1622float2(y[t]);
        acc = fmaf(u.x, v.x, acc);
        acc = fmaf(u.y, v.y, acc);
    }
    return acc;
}

__device__ __forceinline__ float dot16(const uint4& a, const uint4& b, float) {
    const float4 x = *reinterpret_cast<const float4*>(&a);
    const float4 y = *reinterpret_cast<const float4*>(&b);
    return fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, x.w * y.w)));
}

template <typename T>
__global__ void __launch_bounds__(256) route_kernel(const uint4* __restrict__ h,
                                                    const uint4* __restrict__ w, float bias,
                                                    int64_t tokens, int nvec,
                                                    float* __restrict__ logits,
                                                    uint8_t* __restrict__ gate) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t t = warp0; t < tokens; t += nwarps) {
        const uint4* row = h + t * nvec;
        float acc = 0.f;
        int v = lane;
        // four independent 16-byte loads in flight per lane
        for (; v + 96 < nvec; v += 128) {
            const uint4 a0 = __ldcs(row + v), a1 = __ldcs(row + v + 32);
            const uint4 a2 = __ldcs(row + v + 64), a3 = __ldcs(row + v + 96);
            acc += dot16(a0, __ldg(w + v), T()) + dot16(a1, __ldg(w + v + 32), T()) +
                   dot16(a2, __ldg(w + v + 64), T()) + dot16(a3, __ldg(w + v + 96), T());
        }
        for (; v < nvec; v += 32) acc += dot16(__ldcs(row + v), __ldg(w + v), T());
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            const float lg = acc + bias;
            logits[t] = lg;
            gate[t] = lg > 0.f ? 1 : 0;
        }
    }
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
