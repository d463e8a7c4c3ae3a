// Router logits by one warp (SwiAttn report, section 2, router design):
// logit_t = <h_t, w> + b, gate_t = 1(logit_t > 0), fp32 accumulate.  The
// hidden rows stream through 16-byte loads, eight per lane and row in flight,
// two rows at a time.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace swi {

__device__ __forceinline__ float route_dot16(const uint4& a, const uint4& b, __nv_bfloat16) {
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

__device__ __forceinline__ float route_dot16(const uint4& a, const uint4& b, float) {
    const float4 x = *reinterpret_cast<const float4*>(&a);
    const float4 y = *reinterpret_cast<const float4*>(&b);
    return fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, x.w * y.w)));
}

template <typename T>
__device__ __forceinline__ void route_token(const uint4* __restrict__ h, const uint4* __restrict__ w,
                                            float bias, int64_t t, int nvec, float* __restrict__ logits,
                                            uint8_t* __restrict__ gate) {
    const int lane = threadIdx.x & 31;
    const uint4* row = h + t * nvec;
    float acc = 0.f;
    int v = lane;
    for (; v + 224 < nvec; v += 256) {
        uint4 a[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) a[u] = __ldcs(row + v + 32 * u);
        float p = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) p += route_dot16(a[u], __ldg(w + v + 32 * u), T());
        acc += p;
    }
    for (; v < nvec; v += 32) acc += route_dot16(__ldcs(row + v), __ldg(w + v), T());
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
        const float lg = acc + bias;
        logits[t] = lg;
        gate[t] = lg > 0.f ? 1 : 0;
    }
}

// Two tokens t0, t1 by one warp: both rows' loads in flight together.
template <typename T>
__device__ __forceinline__ void route_token2(const uint4* __restrict__ h, const uint4* __restrict__ w,
                                             float bias, int64_t t0, int64_t t1, int nvec,
                                             float* __restrict__ logits, uint8_t* __restrict__ gate) {
    const int lane = threadIdx.x & 31;
    const uint4* ra = h + t0 * nvec;
    const uint4* rb = h + t1 * nvec;
    float acc0 = 0.f, acc1 = 0.f;
    int v = lane;
    for (; v + 224 < nvec; v += 256) {
        uint4 a[8], c[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) a[u] = __ldcs(ra + v + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u) c[u] = __ldcs(rb + v + 32 * u);
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 wv = __ldg(w + v + 32 * u);
            p0 += route_dot16(a[u], wv, T());
            p1 += route_dot16(c[u], wv, T());
        }
        acc0 += p0;
        acc1 += p1;
    }
    for (; v < nvec; v += 32) {
        const uint4 wv = __ldg(w + v);
        acc0 += route_dot16(__ldcs(ra + v), wv, T());
        acc1 += route_dot16(__ldcs(rb + v), wv, T());
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        acc0 += __shfl_xor_sync(0xffffffffu, acc0, o);
        acc1 += __shfl_xor_sync(0xffffffffu, acc1, o);
    }
    if (lane == 0) {
        const float l0 = acc0 + bias, l1 = acc1 + bias;
        logits[t0] = l0;
        gate[t0] = l0 > 0.f ? 1 : 0;
        logits[t1] = l1;
        gate[t1] = l1 > 0.f ? 1 : 0;
    }
}

}  // namespace swi
