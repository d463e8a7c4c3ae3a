// fp32 routed attention on CUDA cores, and the per-token epilogues of the
// dual-branch forward.
//
// The fp32 path keeps every operation in fp32 (no tf32 tensor-core rounding)
// so that it matches the fp64 definition to ~1e-6.  One warp owns one
// (batch, row, head); keys are visited one at a time with an online softmax.
// Key range per row (SwiAttn report, section 2; SWA window per the weimeta.cn
// glossary): routed [0, i], window [max(0, i-W+1), i], plus for a window row
// the global anchors [0, min(S, i-W+1)) (the glossary's 全局锚点).

#include "swiattn_internal.h"

#include <cuda_bf16.h>
#include <math.h>

namespace swi {
namespace {

template <int D>
__global__ void __launch_bounds__(128) simt_attention_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const uint8_t* __restrict__ gate, int force, float* __restrict__ o, float* __restrict__ lse,
    int B, int N, int Hq, int Hkv, int W, int S, float scale) {
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= (int64_t)B * N * Hq) return;
    const int h = (int)(row % Hq);
    const int64_t bi = row / Hq;
    const int i = (int)(bi % N);
    const int b = (int)(bi / N);
    const int kvh = h / (Hq / Hkv);
    const bool routed = force >= 0 ? force != 0 : gate[(size_t)b * N + i] != 0;
    const int lo = routed ? 0 : max(0, i - W + 1);
    const int na = min(S, lo);   // anchors below the window (0 for routed rows)

    float qv[PER], acc[PER];
#pragma unroll
    for (int t = 0; t < PER; ++t) {
        qv[t] = q[row * D + lane + 32 * t];
        acc[t] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const float* kb = k + ((size_t)b * N * Hkv + kvh) * D;
    const float* vb = v + ((size_t)b * N * Hkv + kvh) * D;
    for (int jj = 0; jj < na + (i - lo + 1); ++jj) {
        const int j = jj < na ? jj : lo + (jj - na);
        const float* kj = kb + (size_t)j * Hkv * D;
        float part = 0.f;
#pragma unroll
        for (int t = 0; t < PER; ++t) part = fmaf(qv[t], kj[lane + 32 * t], part);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        const float s = part * scale;
        const float mn = fmaxf(m, s);
        const float corr = expf(m - mn);   // m = -inf on the first key -> 0
        const float p = expf(s - mn);
        l = l * corr + p;
        const float* vj = vb + (size_t)j * Hkv * D;
#pragma unroll
        for (int t = 0; t < PER; ++t) acc[t] = fmaf(p, vj[lane + 32 * t], acc[t] * corr);
        m = mn;
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int t = 0; t < PER; ++t) o[row * D + lane + 32 * t] = acc[t] * inv;
    if (lse && lane == 0) lse[row] = m + logf(l);
}

__device__ __forceinline__ float softplus_f(float x) {
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

// fp32 dual branch: mse over all heads from the fp32 outputs, then gamma, the
// regulariser and the gated output.  One warp per token.
__global__ void __launch_bounds__(128) dual_epilogue_f32_kernel(
    const float* __restrict__ of, const float* __restrict__ os, const float* __restrict__ logits,
    const float* __restrict__ nll, float* __restrict__ og, float* __restrict__ mse,
    float* __restrict__ gamma, float* __restrict__ reg, int BN, int HD, float gb, float eps,
    float alpha, const float* __restrict__ lf, const float* __restrict__ ls,
    float* __restrict__ lg, int Hq) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (t >= BN) return;
    const bool full = logits[t] > 0.f;
    float acc = 0.f;
    for (int c = lane; c < HD; c += 32) {
        const float a = of[t * HD + c], s = os[t * HD + c];
        const float dl = a - s;
        acc = fmaf(dl, dl, acc);
        if (og) og[t * HD + c] = full ? a : s;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
        const float g = gb / (eps + nll[t] + alpha * acc);
        mse[t] = acc;
        gamma[t] = g;
        reg[t] = g * softplus_f(logits[t]);
    }
    if (lg)
        for (int h = lane; h < Hq; h += 32) lg[t * Hq + h] = full ? lf[t * Hq + h] : ls[t * Hq + h];
}

// bf16 dual branch: per-(token, head) squared distances come from the tensor-
// core kernel; sum over heads in a fixed order, then gamma and the regulariser.
__global__ void dual_epilogue_parts_kernel(const float* __restrict__ part,
                                           const float* __restrict__ logits,
                                           const float* __restrict__ nll, float* __restrict__ mse,
                                           float* __restrict__ gamma, float* __restrict__ reg,
                                           int BN, int Hq, float gb, float eps, float alpha) {
    // A programmatic dependent launch of the dual-branch kernel: the partial
    // sums are read after its grid completes.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= BN) return;
    float acc = 0.f;
    for (int h = 0; h < Hq; ++h) acc += part[t * Hq + h];
    const float g = gb / (eps + nll[t] + alpha * acc);
    mse[t] = acc;
    gamma[t] = g;
    reg[t] = g * softplus_f(logits[t]);
}

}  // namespace

cudaError_t launch_simt_attention(const void* q, const void* k, const void* v,
                                  const uint8_t* gate, int force, void* o, float* lse, int B,
                                  int N, int Hq, int Hkv, int d, int W, int S, float scale,
                                  int dtype, cudaStream_t s) {
    if (dtype != 0) return cudaErrorInvalidValue;
    const int64_t rows = (int64_t)B * N * Hq;
    const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
    const float* qf = static_cast<const float*>(q);
    const float* kf = static_cast<const float*>(k);
    const float* vf = static_cast<const float*>(v);
    float* of = static_cast<float*>(o);
    if (d == 64)
        simt_attention_kernel<64><<<blocks, 128, 0, s>>>(qf, kf, vf, gate, force, of, lse, B, N, Hq,
                                                         Hkv, W, S, scale);
    else if (d == 128)
        simt_attention_kernel<128><<<blocks, 128, 0, s>>>(qf, kf, vf, gate, force, of, lse, B, N,
                                                          Hq, Hkv, W, S, scale);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_dual_epilogue_f32(const float* o_full, const float* o_swa,
                                     const float* logits, const float* nll, float* o_gated,
                                     const float* lse_full, const float* lse_swa, float* lse_gated,
                                     float* mse, float* gamma, float* reg, int B, int N, int Hq,
                                     int d, float gamma_base, float eps, float alpha,
                                     cudaStream_t s) {
    const int BN = B * N;
    dual_epilogue_f32_kernel<<<(BN + 3) / 4, 128, 0, s>>>(o_full, o_swa, logits, nll, o_gated, mse,
                                                          gamma, reg, BN, Hq * d, gamma_base, eps,
                                                          alpha, lse_full, lse_swa, lse_gated, Hq);
    return cudaGetLastError();
}

cudaError_t launch_dual_epilogue_parts(const float* mse_part, const float* logits,
                                       const float* nll, float* mse, float* gamma, float* reg,
                                       int B, int N, int Hq, float gamma_base, float eps,
                                       float alpha, cudaStream_t s) {
    const int BN = B * N;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((BN + 255) / 256);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, dual_epilogue_parts_kernel, mse_part, logits,
                                             nll, mse, gamma, reg, BN, Hq, gamma_base, eps, alpha);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace swi
