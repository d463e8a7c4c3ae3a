// fp32 backward of routed attention on CUDA cores, and the router backward.
//
// Attention (dtype fp32, d in {64, 128}): the row-stationary pass gives dq,
// the key-stationary pass dk and dv; one warp per row (or key), lane holds
// d/32 consecutive elements.  Same chain rule as the tensor-core kernels:
//   p_ij = exp(scale q_i.k_j - lse_i),  dS_ij = p_ij (dO_i.v_j - D_i),
//   D_i = dO_i.O_i.
// Router (SwiAttn report, section 2): the straight-through gate passes
// d sigma / d logit = s (1 - s), s = sigmoid(logit); with O = sigma O_FULL +
// (1 - sigma) O_SWA the gate receives dO.(O_FULL - O_SWA); the regulariser
// gamma * softplus(logit) adds gamma * s (gamma is a coefficient).  Then the
// linear router logit = h.w + b gives dh = d_logit w, dw = sum d_logit h,
// db = sum d_logit (fixed-order reductions).

#include "swiattn_internal.h"
#include "swiattn.h"

#include <cuda_bf16.h>
#include <math.h>

namespace swi {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
__device__ __forceinline__ void load_row(const float* src, int lane, float* r) {
    constexpr int E = D / 32;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        const float2 v = reinterpret_cast<const float2*>(src + lane * E)[e / 2];
        r[e] = v.x;
        r[e + 1] = v.y;
    }
}

template <int D>
__device__ __forceinline__ float dot_row(const float* a, const float* b) {
    constexpr int E = D / 32;
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc += a[e] * b[e];
    return warp_sum(acc);
}

// D[b,i,h] = <dO, O>.
template <int D>
__global__ void __launch_bounds__(256) simt_rowdot_kernel(const float* __restrict__ o,
                                                          const float* __restrict__ d_o,
                                                          size_t rows, float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const size_t w = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (w >= rows) return;
    float a[D / 32], b[D / 32];
    load_row<D>(o + w * D, lane, a);
    load_row<D>(d_o + w * D, lane, b);
    const float s = dot_row<D>(a, b);
    if (lane == 0) out[w] = s;
}

// dq: one warp per (b, i, h) over the row's visited keys.
template <int D>
__global__ void __launch_bounds__(256) simt_bwd_dq_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const uint8_t* __restrict__ gate, const float* __restrict__ lse, const float* __restrict__ d_o,
    const float* __restrict__ Drow, float* __restrict__ dq, int B, int N, int Hq, int Hkv, int W,
    float scale) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const size_t row = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= (size_t)B * N * Hq) return;
    const int h = (int)(row % Hq);
    const int i = (int)((row / Hq) % N), b = (int)(row / ((size_t)Hq * N));
    const int kvh = h / (Hq / Hkv);
    const int lo = gate[(size_t)b * N + i] ? 0 : max(0, i - W + 1);
    float qr[E], dor[E], acc[E], kr[E], vr[E];
    load_row<D>(q + row * D, lane, qr);
    load_row<D>(d_o + row * D, lane, dor);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const float L = lse[row], Dv = Drow[row];
    for (int j = lo; j <= i; ++j) {
        const size_t kr_off = (((size_t)b * N + j) * Hkv + kvh) * D;
        load_row<D>(k + kr_off, lane, kr);
        load_row<D>(v + kr_off, lane, vr);
        const float p = expf(scale * dot_row<D>(qr, kr) - L);
        const float ds = p * (dot_row<D>(dor, vr) - Dv);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += ds * kr[e];
    }
#pragma unroll
    for (int e = 0; e < E; e += 2)
        reinterpret_cast<float2*>(dq + row * D + lane * E)[e / 2] =
            make_float2(scale * acc[e], scale * acc[e + 1]);
}

// dk, dv: one warp per (b, j, kv head) over the rows of the group that see
// key j: every row i in [j, j+W-1], and routed rows beyond.
template <int D>
__global__ void __launch_bounds__(256) simt_bwd_dkdv_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const uint8_t* __restrict__ gate, const float* __restrict__ lse, const float* __restrict__ d_o,
    const float* __restrict__ Drow, float* __restrict__ dk, float* __restrict__ dv, int B, int N,
    int Hq, int Hkv, int W, float scale) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const size_t key = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (key >= (size_t)B * N * Hkv) return;
    const int kvh = (int)(key % Hkv);
    const int j = (int)((key / Hkv) % N), b = (int)(key / ((size_t)Hkv * N));
    const int G = Hq / Hkv;
    float kr[E], vr[E], ak[E], av[E], qr[E], dor[E];
    load_row<D>(k + key * D, lane, kr);
    load_row<D>(v + key * D, lane, vr);
#pragma unroll
    for (int e = 0; e < E; ++e) ak[e] = av[e] = 0.f;
    for (int i = j; i < N; ++i) {
        if (i > j + W - 1 && !gate[(size_t)b * N + i]) continue;
        for (int g = 0; g < G; ++g) {
            const size_t row = ((size_t)b * N + i) * Hq + kvh * G + g;
            load_row<D>(q + row * D, lane, qr);
            load_row<D>(d_o + row * D, lane, dor);
            const float p = expf(scale * dot_row<D>(qr, kr) - lse[row]);
            const float ds = p * (dot_row<D>(dor, vr) - Drow[row]);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ak[e] += ds * qr[e];
                av[e] += p * dor[e];
            }
        }
    }
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        reinterpret_cast<float2*>(dk + key * D + lane * E)[e / 2] =
            make_float2(scale * ak[e], scale * ak[e + 1]);
        reinterpret_cast<float2*>(dv + key * D + lane * E)[e / 2] = make_float2(av[e], av[e + 1]);
    }
}

// ------------------------------------------------------------- router ------
template <typename T>
__device__ __forceinline__ void load8(const T* src, float* f);
template <>
__device__ __forceinline__ void load8<float>(const float* src, float* f) {
    const float4 a = reinterpret_cast<const float4*>(src)[0];
    const float4 b = reinterpret_cast<const float4*>(src)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* src, float* f) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float2 x = __bfloat1622float2(p[t]);
        f[2 * t] = x.x;
        f[2 * t + 1] = x.y;
    }
}
template <typename T>
__device__ __forceinline__ void store8(T* dst, const float* f);
template <>
__device__ __forceinline__ void store8<float>(float* dst, const float* f) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const float* f) {
    uint4 u;
    __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int t = 0; t < 4; ++t) p[t] = __floats2bfloat162_rn(f[2 * t], f[2 * t + 1]);
    *reinterpret_cast<uint4*>(dst) = u;
}

// d_logits: one warp per token over its hd outputs (8 elements per step).
template <typename T>
__global__ void __launch_bounds__(256) route_bwd_logit_kernel(
    const float* __restrict__ logits, const T* __restrict__ of, const T* __restrict__ os,
    const T* __restrict__ dout, const float* __restrict__ gamma, const float* __restrict__ d_reg,
    int64_t tokens, int hd, float* __restrict__ d_logits) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= tokens) return;
    float acc = 0.f;
    for (int c = lane * 8; c < hd; c += 256) {
        float a[8], b[8], g[8];
        load8<T>(of + t * hd + c, a);
        load8<T>(os + t * hd + c, b);
        load8<T>(dout + t * hd + c, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc += g[e] * (a[e] - b[e]);
    }
    acc = warp_sum(acc);
    if (lane == 0) {
        const float s = 1.f / (1.f + expf(-logits[t]));
        float dl = s * (1.f - s) * acc;
        if (d_reg) dl += d_reg[t] * gamma[t] * s;
        d_logits[t] = dl;
    }
}

constexpr int kRouteChunk = 64;   // tokens per block of the dh/dw pass

// dh = d_logit * w and per-chunk partial sums of d_logit * h (one block per
// chunk of kRouteChunk tokens; threads stride over 8-column groups).  The
// h rows of kRouteUnroll tokens are loaded before any is used, so that many
// loads are in flight per thread; the sums still run in token order.
constexpr int kRouteUnroll = 8;

template <typename T>
__global__ void __launch_bounds__(256) route_bwd_dh_kernel(
    const T* __restrict__ h, const T* __restrict__ w, const float* __restrict__ d_logits,
    int64_t tokens, int d_model, T* __restrict__ dh, float* __restrict__ part) {
    const int64_t t0 = (int64_t)blockIdx.x * kRouteChunk;
    const int64_t t1 = min(tokens, t0 + kRouteChunk);
    for (int c = threadIdx.x * 8; c < d_model; c += blockDim.x * 8) {
        float wv[8], acc[8];
        load8<T>(w + c, wv);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int64_t tb = t0; tb < t1; tb += kRouteUnroll) {
            float hv[kRouteUnroll][8], dl[kRouteUnroll];
#pragma unroll
            for (int u = 0; u < kRouteUnroll; ++u) {
                const int64_t t = min(tb + u, t1 - 1);   // clamp: duplicates are not used below
                dl[u] = d_logits[t];
                if (part) load8<T>(h + t * d_model + c, hv[u]);
            }
#pragma unroll
            for (int u = 0; u < kRouteUnroll; ++u) {
                if (tb + u >= t1) break;
                if (part) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] += dl[u] * hv[u][e];
                }
                if (dh) {
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = dl[u] * wv[e];
                    store8<T>(dh + (tb + u) * d_model + c, o);
                }
            }
        }
        if (part) store8<float>(part + (int64_t)blockIdx.x * d_model + c, acc);
    }
}

// dw[c] = sum over chunks of the partials: a block takes 32 columns and warp
// w sums chunks w, w+32, w+64, ... for its lane's column, then the 32 warp
// sums are added in warp order (a fixed order, so dw is bitwise repeatable).
// db = sum d_logits (the last block, fixed-order tree).
constexpr int kReduceCols = 32;
constexpr int kReduceWarps = 32;

__global__ void __launch_bounds__(kReduceWarps * 32) route_bwd_reduce_kernel(
    const float* __restrict__ part, int64_t chunks, int d_model, const float* __restrict__ d_logits,
    int64_t tokens, float* __restrict__ dw, float* __restrict__ db) {
    __shared__ float wsum[kReduceWarps][kReduceCols];
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    const int c = blockIdx.x * kReduceCols + lane;
    const bool last = blockIdx.x == gridDim.x - 1;
    const bool do_dw = dw && part && c - lane < d_model;
    if (do_dw) {
        float acc = 0.f;
        if (c < d_model) {
#pragma unroll 8
            for (int64_t k = wp; k < chunks; k += kReduceWarps) acc += part[k * d_model + c];
        }
        wsum[wp][lane] = acc;
    }
    __syncthreads();
    if (do_dw && wp == 0 && c < d_model) {
        float t = 0.f;
#pragma unroll
        for (int u = 0; u < kReduceWarps; ++u) t += wsum[u][lane];
        dw[c] = t;
    }
    if (db && last) {
        __shared__ float red[kReduceWarps * 32];
        float acc = 0.f;
#pragma unroll 8
        for (int64_t t = threadIdx.x; t < tokens; t += blockDim.x) acc += d_logits[t];
        red[threadIdx.x] = acc;
        __syncthreads();
        for (int s = blockDim.x / 2; s > 0; s >>= 1) {
            if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
            __syncthreads();
        }
        if (threadIdx.x == 0) *db = red[0];
    }
}

template <typename T>
cudaError_t route_backward_t(const void* h, const void* w, const float* logits, const void* o_full,
                             const void* o_swa, const void* d_o, const float* gamma,
                             const float* d_reg, int64_t tokens, int hd, int d_model,
                             float* d_logits, void* dh, float* dw, float* db, float* ws,
                             cudaStream_t s) {
    const unsigned blocks = static_cast<unsigned>((tokens + 7) / 8);
    route_bwd_logit_kernel<T><<<blocks, 256, 0, s>>>(
        logits, static_cast<const T*>(o_full), static_cast<const T*>(o_swa),
        static_cast<const T*>(d_o), gamma, d_reg, tokens, hd, d_logits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || (!dh && !dw && !db)) return e;
    const int64_t chunks = route_bwd_chunks(tokens);
    if (dh || dw) {
        route_bwd_dh_kernel<T><<<static_cast<unsigned>(chunks), 256, 0, s>>>(
            static_cast<const T*>(h), static_cast<const T*>(w), d_logits, tokens, d_model,
            static_cast<T*>(dh), dw ? ws : nullptr);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (dw || db) {
        // One block per 32 columns of dw, and one more for db.
        const int blocks_r = (dw ? (d_model + kReduceCols - 1) / kReduceCols : 0) + 1;
        route_bwd_reduce_kernel<<<blocks_r, kReduceWarps * 32, 0, s>>>(
            ws, chunks, d_model, d_logits, tokens, dw, db);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace

cudaError_t launch_simt_backward(const float* q, const float* k, const float* v,
                                 const uint8_t* gate, const float* o, const float* lse,
                                 const float* d_o, float* dq, float* dk, float* dv, int B, int N,
                                 int Hq, int Hkv, int d, int W, float scale, float* ws,
                                 cudaStream_t s) {
    const size_t rows = (size_t)B * N * Hq, keys = (size_t)B * N * Hkv;
    const unsigned rb = static_cast<unsigned>((rows + 7) / 8), kb = static_cast<unsigned>((keys + 7) / 8);
    if (d == 64) {
        simt_rowdot_kernel<64><<<rb, 256, 0, s>>>(o, d_o, rows, ws);
        simt_bwd_dq_kernel<64><<<rb, 256, 0, s>>>(q, k, v, gate, lse, d_o, ws, dq, B, N, Hq, Hkv, W, scale);
        simt_bwd_dkdv_kernel<64><<<kb, 256, 0, s>>>(q, k, v, gate, lse, d_o, ws, dk, dv, B, N, Hq, Hkv, W, scale);
    } else {
        simt_rowdot_kernel<128><<<rb, 256, 0, s>>>(o, d_o, rows, ws);
        simt_bwd_dq_kernel<128><<<rb, 256, 0, s>>>(q, k, v, gate, lse, d_o, ws, dq, B, N, Hq, Hkv, W, scale);
        simt_bwd_dkdv_kernel<128><<<kb, 256, 0, s>>>(q, k, v, gate, lse, d_o, ws, dk, dv, B, N, Hq, Hkv, W, scale);
    }
    return cudaGetLastError();
}

int64_t route_bwd_chunks(int64_t tokens) { return (tokens + kRouteChunk - 1) / kRouteChunk; }

cudaError_t launch_route_backward(const void* h, const void* w, const float* logits,
                                  const void* o_full, const void* o_swa, const void* d_o,
                                  const float* gamma, const float* d_reg, int64_t tokens, int hd,
                                  int d_model, int dtype, float* d_logits, void* dh, float* dw,
                                  float* db, float* ws, cudaStream_t s) {
    if (dtype == SWIATTN_BF16)
        return route_backward_t<__nv_bfloat16>(h, w, logits, o_full, o_swa, d_o, gamma, d_reg,
                                               tokens, hd, d_model, d_logits, dh, dw, db, ws, s);
    return route_backward_t<float>(h, w, logits, o_full, o_swa, d_o, gamma, d_reg, tokens, hd,
                                   d_model, d_logits, dh, dw, db, ws, s);
}

}  // namespace swi
