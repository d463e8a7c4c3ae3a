// Scheduling and per-row statistics of the routed-attention backward.
//
// The gradient of row i flows through the branch its hard gate selected (the
// straight-through gate's forward value is 0/1; SwiAttn report, section 2),
// so the (query, key) pairs of the backward are those of the forward:
// window rows visit [max(0, i-W+1), i], far rows (gate = 1, i >= W) [0, i].
//
// Per row the backward needs D_i = <dO_i, O_i> and the forward's log-sum-exp
// (kept here pre-multiplied by log2 e, for exp2 in the kernels).  Two layouts:
//  - band arrays [B, Hq, Npad] indexed by row i (Npad = N rounded up to 128,
//    zero past N), read by the key-stationary kernel 128 columns at a time;
//  - far arrays [B, Hq, Npad] indexed by compacted far-row position, with
//    the compacted q and dO of far rows ([B, Npad, Hq, 128] bf16) and their
//    row indices, zero-padded to a whole 128-row tile (kNoRow in the index).
// Work lists (cost-sorted, longest first, claimed dynamically):
//  - dK/dV: one item per (b, kv head, 128-key block);
//  - dQ: one item per (b, query head) band tile (skipped when every row of it
//    is a far row) and per (b, query head) far tile.

#include "swiattn_internal.h"

#include <cuda_bf16.h>

namespace swi {
namespace {

constexpr int kBuildThreads = 512;
constexpr int kCostBuckets = 4096;
constexpr int kBucketsPerThread = kCostBuckets / kBuildThreads;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// <a, b> over one 128-element bf16 row, one warp (4 elements per lane).
__device__ __forceinline__ float row_dot_bf16(const __nv_bfloat16* a, const __nv_bfloat16* b,
                                              int lane) {
    const uint2 ua = reinterpret_cast<const uint2*>(a)[lane];
    const uint2 ub = reinterpret_cast<const uint2*>(b)[lane];
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&ua);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&ub);
    const float2 a0 = __bfloat1622float2(pa[0]), a1 = __bfloat1622float2(pa[1]);
    const float2 b0 = __bfloat1622float2(pb[0]), b1 = __bfloat1622float2(pb[1]);
    float acc = a0.x * b0.x + a0.y * b0.y + a1.x * b1.x + a1.y * b1.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

// Band statistics, one warp per (b, i, h) with i < Npad (h fastest, so a
// warp group reads whole contiguous token rows).
__global__ void __launch_bounds__(256) bwd_rowstats_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o,
    const float* __restrict__ lse, int B, int N, int Npad, int Hq, float* __restrict__ d_band,
    float* __restrict__ l_band) {
    const int lane = threadIdx.x & 31;
    const size_t nrows = (size_t)B * Npad * Hq;
    const size_t stride = (size_t)gridDim.x * (blockDim.x >> 5);
    for (size_t w = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < nrows;
         w += stride) {
        const int h = (int)(w % Hq);
        const size_t bi = w / Hq;
        const int i = (int)(bi % Npad), b = (int)(bi / Npad);
        float dd = 0.f, ll = 0.f;
        if (i < N) {
            const size_t row = ((size_t)b * N + i) * Hq + h;
            dd = row_dot_bf16(d_o + row * kHD, o + row * kHD, lane);
            ll = lse[row] * kLog2e;
        }
        if (lane == 0) {
            const size_t dst = ((size_t)b * Hq + h) * Npad + i;
            d_band[dst] = dd;
            l_band[dst] = ll;
        }
    }
}

// Binary search: first position of sorted list[0, n) holding a value >= x.
__device__ __forceinline__ int lower_bound_dev(const int* list, int n, int x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (list[mid] >= x) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// dK/dV item u = ((b * Hkv) + kvh) * NB + kb.
__device__ __forceinline__ BwdItem kv_item(int u, const int* routed_list, const int* routed_count,
                                           int N, int Hq, int Hkv, int W, int NB) {
    BwdItem it;
    it.kind = kBwdKV;
    it.t = u % NB;
    it.h = (u / NB) % Hkv;
    it.b = u / (NB * Hkv);
    const int k0 = it.t * kBN;
    it.a0 = cdiv(min(N, k0 + kBN - 1 + W) - k0, kBM);   // band query tiles
    const int R = routed_count[it.b];
    const int first = lower_bound_dev(routed_list + (size_t)it.b * N, R, k0 + W);
    it.a1 = first < R ? first / kBM : 0;                // far tiles [a1, a2)
    it.a2 = first < R ? cdiv(R, kBM) : 0;
    it.cost = (Hq / Hkv) * (it.a0 + it.a2 - it.a1);
    return it;
}

// dQ item u = b * 2NT + (band tile | NT + far tile); cost 0 = nothing to do.
__device__ __forceinline__ BwdItem q_item(int u, const int* routed_list, const int* routed_count,
                                          const int* tile_prefix, int N, int W, int NT) {
    BwdItem it;
    it.b = u / (2 * NT);
    const int rem = u % (2 * NT);
    it.h = 0;
    it.a2 = 0;
    it.cost = 0;
    if (rem < NT) {
        it.kind = kBwdQBand;
        it.t = rem;
        const int q0 = rem * kBM;
        const int nrows = min(kBM, N - q0);
        const int far_rows = tile_prefix[(size_t)it.b * (NT + 1) + rem + 1] -
                             tile_prefix[(size_t)it.b * (NT + 1) + rem];
        it.a0 = max(0, q0 - W + 1);
        it.a1 = (q0 + nrows - 1 - it.a0) / kBN + 1;
        if (far_rows < nrows) it.cost = it.a1;
    } else {
        it.kind = kBwdQFar;
        it.t = rem - NT;
        const int R = routed_count[it.b];
        it.a0 = 0;
        it.a1 = 0;
        if (it.t * kBM < R) {
            const int last = routed_list[(size_t)it.b * N + min(R, (it.t + 1) * kBM) - 1];
            it.a1 = last / kBN + 1;
            it.cost = it.a1;
        }
    }
    return it;
}

// Counting sort of U candidate items by descending cost into `items` (each
// expanded into `fan` items with h = 0..fan-1 when fan > 1).  One block.
template <typename MakeItem>
__device__ void sort_items(int U, int fan, MakeItem make, BwdItem* items, int* n_out,
                           int* next_out) {
    __shared__ int hist[kCostBuckets];
    __shared__ int warp_tot[32];
    for (int c = threadIdx.x; c < kCostBuckets; c += blockDim.x) hist[c] = 0;
    __syncthreads();
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
        const BwdItem it = make(u);
        if (it.cost > 0) atomicAdd(&hist[min(it.cost, kCostBuckets - 1)], 1);
    }
    __syncthreads();
    // Exclusive offsets in descending cost order; thread t owns the buckets
    // kCostBuckets-1-8t ... kCostBuckets-8-8t.
    int own = 0;
#pragma unroll
    for (int k = 0; k < kBucketsPerThread; ++k)
        own += hist[kCostBuckets - 1 - (threadIdx.x * kBucketsPerThread + k)];
    // block exclusive scan of `own`
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    int run = (w > 0 ? warp_tot[w - 1] : 0) + x - own;
    const int total = warp_tot[nw - 1];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBucketsPerThread; ++k) {
        const int c = kCostBuckets - 1 - (threadIdx.x * kBucketsPerThread + k);
        const int hcount = hist[c];
        hist[c] = run;
        run += hcount;
    }
    __syncthreads();
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
        BwdItem it = make(u);
        if (it.cost <= 0) continue;
        const int pos = atomicAdd(&hist[min(it.cost, kCostBuckets - 1)], 1);
        for (int h = 0; h < fan; ++h) {
            it.h = (fan > 1) ? h : it.h;
            items[(size_t)pos * fan + h] = it;
        }
    }
    if (threadIdx.x == 0) {
        *n_out = total * fan;
        *next_out = 0;   // work counter the kernel claims items from
    }
}

// Block 0: dK/dV list.  Block 1: dQ list.  Other blocks: compaction of far
// rows (q, dO, D, lse, row index), zero-padded to whole 128-row tiles.
__global__ void __launch_bounds__(kBuildThreads) bwd_build_gather_kernel(
    const int* __restrict__ routed_list, const int* __restrict__ routed_count,
    const int* __restrict__ tile_prefix, int B, int N, int Npad, int Hq, int Hkv, int W,
    BwdItem* __restrict__ items_kv, BwdItem* __restrict__ items_q, int* __restrict__ counters,
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ o,
    const float* __restrict__ lse, const __nv_bfloat16* __restrict__ d_o,
    __nv_bfloat16* __restrict__ qc, __nv_bfloat16* __restrict__ doc, float* __restrict__ d_far,
    float* __restrict__ l_far, int* __restrict__ rowidx) {
    const int NT = cdiv(N, kBM);
    if (blockIdx.x == 0) {
        sort_items(
            B * Hkv * NT, 1,
            [&](int u) { return kv_item(u, routed_list, routed_count, N, Hq, Hkv, W, NT); },
            items_kv, &counters[0], &counters[1]);
        return;
    }
    if (blockIdx.x == 1) {
        sort_items(
            B * 2 * NT, Hq,
            [&](int u) { return q_item(u, routed_list, routed_count, tile_prefix, N, W, NT); },
            items_q, &counters[2], &counters[3]);
        return;
    }
    const int lane = threadIdx.x & 31;
    const size_t warps = (size_t)(gridDim.x - 2) * (blockDim.x >> 5);
    const size_t w0 = (size_t)(blockIdx.x - 2) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (int b = 0; b < B; ++b) {
        const int R = routed_count[b];
        const int Rp = cdiv(R, kBM) * kBM;
        for (size_t w = w0; w < (size_t)Rp * Hq; w += warps) {
            const int r = (int)(w / Hq), h = (int)(w % Hq);
            const size_t dst = ((size_t)b * Npad + r) * Hq + h;
            uint2 vq = make_uint2(0u, 0u), vd = make_uint2(0u, 0u);
            float dd = 0.f, ll = 0.f;
            int i = kNoRow;
            if (r < R) {
                i = routed_list[(size_t)b * N + r];
                const size_t src = ((size_t)b * N + i) * Hq + h;
                vq = reinterpret_cast<const uint2*>(q + src * kHD)[lane];
                vd = reinterpret_cast<const uint2*>(d_o + src * kHD)[lane];
                dd = row_dot_bf16(d_o + src * kHD, o + src * kHD, lane);
                ll = lse[src] * kLog2e;
            }
            reinterpret_cast<uint2*>(qc + dst * kHD)[lane] = vq;
            reinterpret_cast<uint2*>(doc + dst * kHD)[lane] = vd;
            if (lane == 0) {
                d_far[((size_t)b * Hq + h) * Npad + r] = dd;
                l_far[((size_t)b * Hq + h) * Npad + r] = ll;
                if (h == 0) rowidx[(size_t)b * Npad + r] = i;
            }
        }
    }
}

}  // namespace

BwdWs bwd_ws_layout(int B, int N, int Hq, int Hkv) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t NT = (static_cast<size_t>(N) + kBM - 1) / kBM;
    BwdWs L;
    L.Npad = static_cast<int>(NT * kBM);
    L.max_kv = static_cast<int>((size_t)B * Hkv * NT);
    L.max_q = static_cast<int>((size_t)B * 2 * NT * Hq);
    const size_t rows = (size_t)B * Hq * L.Npad;
    size_t off = 0;
    L.routed_list = off;
    off = up(off + sizeof(int) * (size_t)B * N);
    L.routed_count = off;
    off = up(off + sizeof(int) * (size_t)B);
    L.tile_prefix = off;
    off = up(off + sizeof(int) * (size_t)B * (NT + 1));
    L.rowidx = off;
    off = up(off + sizeof(int) * (size_t)B * L.Npad);
    L.d_band = off;
    off = up(off + sizeof(float) * rows);
    L.l_band = off;
    off = up(off + sizeof(float) * rows);
    L.d_far = off;
    off = up(off + sizeof(float) * rows);
    L.l_far = off;
    off = up(off + sizeof(float) * rows);
    L.qc = off;
    off = up(off + 2 * rows * kHD);
    L.doc = off;
    off = up(off + 2 * rows * kHD);
    L.counters = off;
    off = up(off + sizeof(int) * 4);
    L.items_kv = off;
    off = up(off + sizeof(BwdItem) * (size_t)L.max_kv);
    L.items_q = off;
    off = up(off + sizeof(BwdItem) * (size_t)L.max_q);
    L.total = off;
    return L;
}

cudaError_t launch_bwd_schedule(const uint8_t* gate, const void* q, const void* o,
                                const float* lse, const void* d_o, int B, int N, int Hq,
                                int Hkv, int W, const BwdWs& L, char* ws, int num_sms,
                                cudaStream_t s) {
    int* list = reinterpret_cast<int*>(ws + L.routed_list);
    int* count = reinterpret_cast<int*>(ws + L.routed_count);
    int* prefix = reinterpret_cast<int*>(ws + L.tile_prefix);
    cudaError_t e = launch_far_scan(gate, B, N, W, list, count, prefix, s);
    if (e != cudaSuccess) return e;
    const auto* ob = static_cast<const __nv_bfloat16*>(o);
    const auto* dob = static_cast<const __nv_bfloat16*>(d_o);
    bwd_rowstats_kernel<<<num_sms * 8, 256, 0, s>>>(ob, dob, lse, B, N, L.Npad, Hq,
                                                    reinterpret_cast<float*>(ws + L.d_band),
                                                    reinterpret_cast<float*>(ws + L.l_band));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_build_gather_kernel<<<2 + num_sms * 2, kBuildThreads, 0, s>>>(
        list, count, prefix, B, N, L.Npad, Hq, Hkv, W,
        reinterpret_cast<BwdItem*>(ws + L.items_kv), reinterpret_cast<BwdItem*>(ws + L.items_q),
        reinterpret_cast<int*>(ws + L.counters), static_cast<const __nv_bfloat16*>(q), ob, lse,
        dob, reinterpret_cast<__nv_bfloat16*>(ws + L.qc),
        reinterpret_cast<__nv_bfloat16*>(ws + L.doc), reinterpret_cast<float*>(ws + L.d_far),
        reinterpret_cast<float*>(ws + L.l_far), reinterpret_cast<int*>(ws + L.rowidx));
    return cudaGetLastError();
}

}  // namespace swi
