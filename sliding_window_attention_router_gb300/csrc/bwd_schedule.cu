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

// <a, b> of 8 bf16 pairs held in two 16-byte words.
__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b) {
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float2 x = __bfloat1622float2(pa[t]), y = __bfloat1622float2(pb[t]);
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
    }
    return acc;
}

// Band statistics.  One warp per token (b, i): its Hq head rows are one
// contiguous run, a row of 128 bf16 being 16 lanes x 16 bytes, so the warp
// covers two rows per step and issues every load of the token before the
// half-warp reductions.
constexpr int kMaxHeadPairs = 8;   // 16 heads per pass; more heads take more passes
__global__ void __launch_bounds__(256) bwd_rowstats_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o,
    const float* __restrict__ lse, int B, int N, int Npad, int Hq, float* __restrict__ d_band,
    float* __restrict__ l_band) {
    const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
    const unsigned tokens = (unsigned)B * (unsigned)Npad;
    const unsigned stride = gridDim.x * (blockDim.x >> 5);
    for (unsigned t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < tokens; t += stride) {
        const int b = (int)(t / (unsigned)Npad), i = (int)(t % (unsigned)Npad);
        const bool in = i < N;
        const size_t row0 = ((size_t)b * N + i) * Hq;   // first head row of the token
        for (int h0 = 0; h0 < Hq; h0 += 2 * kMaxHeadPairs) {
            uint4 va[kMaxHeadPairs], vb[kMaxHeadPairs];
#pragma unroll
            for (int u = 0; u < kMaxHeadPairs; ++u) {
                const int h = h0 + 2 * u + half;
                const bool ok = in && h < Hq;
                va[u] = ok ? reinterpret_cast<const uint4*>(d_o + (row0 + h) * kHD)[sub] : make_uint4(0, 0, 0, 0);
                vb[u] = ok ? reinterpret_cast<const uint4*>(o + (row0 + h) * kHD)[sub] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kMaxHeadPairs; ++u) {
                float acc = dot8_bf16(va[u], vb[u]);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                const int h = h0 + 2 * u + half;
                if (sub == 0 && h < Hq) {
                    const size_t dst = ((size_t)b * Hq + h) * Npad + i;
                    d_band[dst] = acc;
                    l_band[dst] = in ? lse[row0 + h] * kLog2e : 0.f;
                }
            }
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
    const int front = far_front(R);
    const int first = lower_bound_dev(routed_list + (size_t)it.b * N, R, k0 + W);
    it.a1 = first < R ? (first + front) / kBM : 0;      // far tiles [a1, a2)
    it.a2 = first < R ? (R + front) / kBM : 0;
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
        const int front = far_front(R);
        it.a0 = 0;
        it.a1 = 0;
        if (it.t * kBM < R + front) {
            const int last = routed_list[(size_t)it.b * N + min(R, (it.t + 1) * kBM - front) - 1];
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
// rows (q, dO, D, lse, row index), zero-padded to whole 128-row tiles; D and
// lse come from the band statistics (computed before, by row).
__global__ void __launch_bounds__(kBuildThreads) bwd_build_gather_kernel(
    const int* __restrict__ routed_list, const int* __restrict__ routed_count,
    const int* __restrict__ tile_prefix, int B, int N, int Npad, int Hq, int Hkv, int W,
    BwdItem* __restrict__ items_kv, BwdItem* __restrict__ items_q, int* __restrict__ counters,
    const __nv_bfloat16* __restrict__ q, const float* __restrict__ d_band,
    const float* __restrict__ l_band, const __nv_bfloat16* __restrict__ d_o,
    __nv_bfloat16* __restrict__ qc, __nv_bfloat16* __restrict__ doc, float* __restrict__ d_far,
    float* __restrict__ l_far, int* __restrict__ rowidx) {
    // The dK/dV kernel after it is a programmatic dependent launch: its CTAs
    // may start on SMs this grid leaves (they wait for it before reading).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
    // Far rows: half a warp per (compacted row, head), 16 bytes per lane.
    const int lane = threadIdx.x & 31, half = lane >> 4, sub = lane & 15;
    const size_t warps = (size_t)(gridDim.x - 2) * (blockDim.x >> 5);
    const size_t w0 = (size_t)(blockIdx.x - 2) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (int b = 0; b < B; ++b) {
        const int R = routed_count[b];
        const int front = far_front(R);
        const size_t total = (size_t)(R + front) * Hq;   // (position, head) pairs to write
        for (size_t ww = w0; 2 * ww < total; ww += warps) {
            const size_t w = 2 * ww + half;
            const bool live = w < total;
            const int pos = (int)(w / Hq), h = (int)(w % Hq);
            const int r = pos - front;   // compacted far row at this position
            uint4 vq = make_uint4(0u, 0u, 0u, 0u), vd = vq;
            int i = kNoRow;
            float dv = 0.f, lv = 0.f;
            if (live && r >= 0 && r < R) {
                i = routed_list[(size_t)b * N + r];
                const size_t src = ((size_t)b * N + i) * Hq + h;
                vq = reinterpret_cast<const uint4*>(q + src * kHD)[sub];
                vd = reinterpret_cast<const uint4*>(d_o + src * kHD)[sub];
                if (sub == 0) {
                    const size_t stat = ((size_t)b * Hq + h) * Npad + i;
                    dv = d_band[stat];
                    lv = l_band[stat];
                }
            }
            if (live) {
                const size_t dst = ((size_t)b * Npad + pos) * Hq + h;
                reinterpret_cast<uint4*>(qc + dst * kHD)[sub] = vq;
                reinterpret_cast<uint4*>(doc + dst * kHD)[sub] = vd;
                if (sub == 0) {
                    d_far[((size_t)b * Hq + h) * Npad + pos] = dv;
                    l_far[((size_t)b * Hq + h) * Npad + pos] = lv;
                    if (h == 0) rowidx[(size_t)b * Npad + pos] = i;
                }
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
    bwd_rowstats_kernel<<<num_sms * 4, 256, 0, s>>>(ob, dob, lse, B, N, L.Npad, Hq,
                                                    reinterpret_cast<float*>(ws + L.d_band),
                                                    reinterpret_cast<float*>(ws + L.l_band));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_build_gather_kernel<<<2 + num_sms * 2, kBuildThreads, 0, s>>>(
        list, count, prefix, B, N, L.Npad, Hq, Hkv, W,
        reinterpret_cast<BwdItem*>(ws + L.items_kv), reinterpret_cast<BwdItem*>(ws + L.items_q),
        reinterpret_cast<int*>(ws + L.counters), static_cast<const __nv_bfloat16*>(q),
        reinterpret_cast<const float*>(ws + L.d_band), reinterpret_cast<const float*>(ws + L.l_band),
        dob, reinterpret_cast<__nv_bfloat16*>(ws + L.qc),
        reinterpret_cast<__nv_bfloat16*>(ws + L.doc), reinterpret_cast<float*>(ws + L.d_far),
        reinterpret_cast<float*>(ws + L.l_far), reinterpret_cast<int*>(ws + L.rowidx));
    return cudaGetLastError();
}

}  // namespace swi
