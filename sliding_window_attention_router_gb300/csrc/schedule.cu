// Gate-driven scheduling for the routed prefill (one launch).
//
// A row i of batch b is a "far" row when its gate routes it to full attention
// and i >= W (for i < W its full range [0, i] equals its window).  Far rows
// are compacted (ascending i) so that 128 of them share one query tile that
// walks keys [0, max i]; every other row is served by the 128-row band tile
// that holds it, which walks only the window keys.  Work items are pairs of
// such tiles (256 rows, one head).  For the persistent attention kernel the
// list holds the far pairs head by head, longest first within a head (cost
// in key blocks), then the band pairs in row order, the heads of a pair
// adjacent.  A far pair too long for the balance of the launch is listed as
// its two tiles instead (see plan_block).

#include "route_gemv.cuh"
#include "swiattn_internal.h"

#include <cuda_bf16.h>
#include <climits>

namespace swi {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kCostBuckets = 4096;

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Block-wide exclusive scan of one value per thread; *total receives the sum.
// Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_tot[lane] = t;   // inclusive totals per warp
    }
    __syncthreads();
    const int excl = (w > 0 ? warp_tot[w - 1] : 0) + x - v;
    *total = warp_tot[nwarps - 1];
    __syncthreads();
    return excl;
}

// One CTA per batch, one pass: each thread counts the far-row flags of a
// contiguous chunk (all its gate loads in flight), one block scan, then each
// thread writes its far rows and the per-tile prefix counts of its chunk.
__global__ void __launch_bounds__(kScanThreads) scan_far_rows_kernel(
    const uint8_t* __restrict__ gate, int N, int W, int* __restrict__ routed_list,
    int* __restrict__ routed_count, int* __restrict__ tile_prefix) {
    __shared__ int warp_tot[32];
    const int b = blockIdx.x;
    const int NT = cdiv(N, kBM);
    const int C = cdiv(N, kScanThreads);
    const int i0 = min(N, threadIdx.x * C), i1 = min(N, i0 + C);
    const uint8_t* g = gate + (size_t)b * N;
    int cnt = 0;
#pragma unroll 8
    for (int i = i0; i < i1; ++i) cnt += (i >= W && g[i] != 0) ? 1 : 0;
    int total;
    int run = block_exclusive_scan(cnt, warp_tot, &total);
    int* list = routed_list + (size_t)b * N;
    int* pre = tile_prefix + (size_t)b * (NT + 1);
    for (int i = i0; i < i1; ++i) {
        if ((i % kBM) == 0) pre[i / kBM] = run;
        if (i >= W && g[i] != 0) list[run++] = i;
    }
    if (threadIdx.x == 0) {
        routed_count[b] = total;
        pre[NT] = total;
    }
}

// Key blocks a 128-row band tile starting at row r0 walks, or 0 when it has
// no row to write (out of range, or every row is a far row).
__device__ __forceinline__ int band_tile_blocks(int b, int r0, int kv0, const int* tile_prefix,
                                                int N, int W, int NT) {
    const int nrows = min(kBM, N - r0);
    if (nrows <= 0) return 0;
    const int t = r0 / kBM;
    const int far_rows = tile_prefix[(size_t)b * (NT + 1) + t + 1] -
                         tile_prefix[(size_t)b * (NT + 1) + t];
    if (far_rows >= nrows) return 0;
    const int lo_key = max(0, r0 - W + 1);
    return (r0 + nrows - 1 - kv0) / kBN - (lo_key - kv0) / kBN + 1;
}

// Anchor key blocks a band tile starting at row r0 adds (window rows see the
// first S keys too): keys [0, min(S, last row - W + 1)).
__device__ __forceinline__ int anchor_blocks(int r0, int N, int W, int S) {
    const int last = min(N, r0 + kBM) - 1;
    const int hi = min(S - 1, last - W);
    return (S > 0 && last >= r0 && hi >= 0) ? hi / kBN + 1 : 0;
}

// Key blocks of far pair `pair` of batch b (both tiles): a far tile walks
// keys [0, last row]; far_last holds each far tile's last row (-1 past the
// last far tile).
__device__ __forceinline__ int far_tile_cost(int b, int k, const int* far_last, int NT) {
    const int r = k < NT ? far_last[(size_t)b * NT + k] : -1;
    return r >= 0 ? r / kBN + 1 : 0;
}

__device__ __forceinline__ int far_pair_cost(int b, int pair, const int* far_last, int NT) {
    int cost = 0;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int k = 2 * pair + x;
        const int r = k < NT ? far_last[(size_t)b * NT + k] : -1;
        if (r >= 0) cost += r / kBN + 1;
    }
    return cost;
}

// Key blocks of band pair `pair` of batch b (both tiles, anchor runs
// included), or 0 when neither tile has a row to write.
__device__ __forceinline__ int band_pair_cost(int b, int pair, const int* tile_prefix, int N,
                                              int W, int S, int NT) {
    const int q0 = pair * 2 * kBM;
    const int kv0 = max(0, q0 - W + 1);
    const int na = max(anchor_blocks(q0, N, W, S), anchor_blocks(q0 + kBM, N, W, S));
    const int cost = band_tile_blocks(b, q0, kv0, tile_prefix, N, W, NT) +
                     band_tile_blocks(b, q0 + kBM, kv0, tile_prefix, N, W, NT);
    return cost > 0 ? cost + 2 * na : 0;
}

// Gate bytes i .. i+15 of one batch row (zero where i+u >= N).  A whole
// in-range group is one 16-byte load when the row start is 16-byte aligned.
// The loads bypass L1: in the fused router + schedule kernel other CTAs wrote
// the gates moments before.
__device__ __forceinline__ uint4 load_gates16(const uint8_t* g, int i, int N, bool vec) {
    if (vec && i + 16 <= N) return __ldcg(reinterpret_cast<const uint4*>(g + i));
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int u = 0; u < 16; ++u)
        if (i + u < N)
            w[u >> 2] |= static_cast<uint32_t>(__ldcg(g + i + u) != 0 ? 1u : 0u) << (8 * (u & 3));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ bool gate_byte(const uint4& v, int u) {
    const uint32_t w = u < 4 ? v.x : u < 8 ? v.y : u < 12 ? v.z : v.w;
    return ((w >> (8 * (u & 3))) & 0xFFu) != 0;
}

// The whole prefill schedule in one CTA, in two passes with one global round
// trip each.  Pass 1, per batch: each thread counts the far rows of a
// contiguous chunk of rows (a multiple of 16, so 16-byte gate groups never
// straddle two threads), one block scan, then each thread writes its far rows
// (ascending i), the prefix counts of the 128-row tiles that start in its
// chunk, and the last row of each far tile that ends in its chunk.  Pass 2:
// the cost of every pair from those per-tile values, a histogram of the far
// costs and the number of busy band pairs of each thread's run, one scan of
// both, then the work list, Hq items per 256-row pair (one per query head):
// far pairs sorted by descending cost, then band pairs in order; and the
// reset of the attention kernel's work counter.  Far queries are not copied
// here: the attention kernel gathers them by row index when it loads a far
// tile.
constexpr int kPlanThreads = 1024;
constexpr int kBucketsPerThread = kCostBuckets / kPlanThreads;
// Per-tile values (far tiles' last rows, tile prefixes) of batches with up to
// this many tiles in all are also kept in shared memory for pass 2.
constexpr int kTileCache = 2048;
// With up to this many pairs, each item's pair is first noted in shared
// memory by list position, and the items are then written by consecutive
// threads in list order (coalesced) instead of by the thread of their pair.
constexpr int kPairCache = 1024;

// Block-wide exclusive scan of two values per thread at once; every thread
// of the block must call it.
__device__ __forceinline__ int2 block_exclusive_scan2(int2 v, int2* warp_tot, int2* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int2 x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yx = __shfl_up_sync(0xffffffffu, x.x, o);
        const int yy = __shfl_up_sync(0xffffffffu, x.y, o);
        if (lane >= o) {
            x.x += yx;
            x.y += yy;
        }
    }
    if (lane == 31) warp_tot[w] = x;
    __syncthreads();
    if (w == 0) {
        int2 t = lane < nwarps ? warp_tot[lane] : make_int2(0, 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yx = __shfl_up_sync(0xffffffffu, t.x, o);
            const int yy = __shfl_up_sync(0xffffffffu, t.y, o);
            if (lane >= o) {
                t.x += yx;
                t.y += yy;
            }
        }
        warp_tot[lane] = t;   // inclusive totals per warp
    }
    __syncthreads();
    const int2 before = w > 0 ? warp_tot[w - 1] : make_int2(0, 0);
    *total = warp_tot[nwarps - 1];
    __syncthreads();
    return make_int2(before.x + x.x - v.x, before.y + x.y - v.y);
}

// Every thread of a kPlanThreads-thread block calls it.
__device__ void plan_block(const uint8_t* __restrict__ gate, int B, int N, int Hq, int W, int S,
                           int grid, int* __restrict__ routed_list, int* __restrict__ routed_count,
                           int* __restrict__ tile_prefix, int* __restrict__ far_last,
                           WorkItem* __restrict__ items, int* __restrict__ n_items) {
    __shared__ int hist[kCostBuckets];
    __shared__ int warp_tot[32];
    __shared__ int2 warp_tot2[32];
    __shared__ int s_last[kTileCache];
    __shared__ int s_pre[kTileCache];
    __shared__ int s_at[2 * kPairCache];   // far position -> pair | kind << 24; band position -> order index
    __shared__ float3 s_cost[32];   // per warp: far, band pair cost sums, largest far pair cost
    const int NT = cdiv(N, kBM);
    const int NP = cdiv(N, 2 * kBM);
    const bool cached = (int64_t)B * (NT + 1) <= kTileCache;
    const int C = cdiv(cdiv(N, kPlanThreads), 16) * 16;
    for (int c = threadIdx.x; c < kCostBuckets; c += blockDim.x) hist[c] = 0;
    for (int b = 0; b < B; ++b) {
        const uint8_t* g = gate + (size_t)b * N;
        const bool vec = (reinterpret_cast<uintptr_t>(g) & 15u) == 0;
        const int i0 = min(N, static_cast<int>(threadIdx.x) * C), i1 = min(N, i0 + C);
        int cnt = 0;
        for (int i = i0; i < i1; i += 16) {
            const uint4 v = load_gates16(g, i, N, vec);
#pragma unroll
            for (int u = 0; u < 16; ++u) cnt += (i + u >= W && i + u < i1 && gate_byte(v, u)) ? 1 : 0;
        }
        int total;
        int run = block_exclusive_scan(cnt, warp_tot, &total);
        int* list = routed_list + (size_t)b * N;
        int* pre = tile_prefix + (size_t)b * (NT + 1);
        int* last = (cached ? s_last : far_last) + (size_t)b * NT;
        // Far tile t holds compacted rows [128 t - front, 128 t - front + 128):
        // the first one takes the remainder (the attention kernel derives the
        // same offset from the count).
        const int front = far_front(total);
        for (int i = i0; i < i1; i += 16) {
            const uint4 v = load_gates16(g, i, N, vec);
            if ((i % kBM) == 0) {   // 16 divides 128: tile starts begin groups
                pre[i / kBM] = run;
                if (cached) s_pre[b * (NT + 1) + i / kBM] = run;
            }
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (i + u >= W && i + u < i1 && gate_byte(v, u)) {
                    if ((run + front) % kBM == kBM - 1 || run == total - 1) last[(run + front) / kBM] = i + u;
                    list[run++] = i + u;
                }
        }
        // Far tiles past the last one hold no rows.
        for (int k = cdiv(total + front, kBM) + threadIdx.x; k < NT; k += blockDim.x) last[k] = -1;
        if (threadIdx.x == 0) {
            routed_count[b] = total;
            pre[NT] = total;
            if (cached) s_pre[b * (NT + 1) + NT] = total;
        }
    }
    __syncthreads();   // the per-tile values above are read below
    const int* fl = cached ? s_last : far_last;
    const int* tp = cached ? s_pre : tile_prefix;

    // Far pairs: counting sort by descending cost (they cost up to N / 128
    // key blocks per tile, so longest first matters for the balance of the
    // persistent kernel), listed head by head: the CTAs that take them at the
    // same time then walk the K/V prefix of few heads, from key 0 up, and
    // share it in L2 (with the heads interleaved, the 32K workload read
    // 2.2x its algorithmic bytes from HBM; head by head, 1.45x).
    const int U = B * NP;
    int far_sum = 0, far_max = 0;
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
        const int cost = far_pair_cost(u / NP, u % NP, fl, NT);
        if (cost > 0) atomicAdd(&hist[min(cost, kCostBuckets - 1)], 1);
        far_sum += cost;
        far_max = max(far_max, cost);
    }

    // Band pairs follow, in (batch, pair) order with the heads of a pair
    // adjacent: their costs are nearly equal (the window and one tile), and
    // the CTAs that run them at the same time then walk overlapping windows
    // of the same heads, which L2 serves.  The pairs whose window reaches
    // back past row 0 (the first E of each batch) cost fewer key blocks the
    // earlier they start; they close the list, latest first, so the last
    // items claimed are the shortest.  Each thread takes a contiguous run of
    // the order; the scan below places the runs.
    const int E = min(NP, cdiv(W - 1, 2 * kBM));
    const int UF = B * (NP - E);
    auto band_at = [&](int v, int& b, int& pair) {
        if (v < UF) {
            b = v / (NP - E);
            pair = E + v % (NP - E);
        } else {
            b = (v - UF) / E;
            pair = E - 1 - (v - UF) % E;
        }
    };
    const int CB = cdiv(U, kPlanThreads);
    const int v0 = min(U, static_cast<int>(threadIdx.x) * CB), v1 = min(U, v0 + CB);
    int nb = 0, band_sum = 0;
    for (int v = v0; v < v1; ++v) {
        int b, pair;
        band_at(v, b, pair);
        const int cost = band_pair_cost(b, pair, tp, N, W, S, NT);
        nb += cost > 0;
        band_sum += cost;
    }
    // Cost sums and the largest far pair cost: warp shuffles, then one slot
    // per warp (one shared address taking an atomic from every thread cost
    // ~6000 cycles here), read by every thread after the barrier.
    {
        float fs = static_cast<float>(far_sum), bs = static_cast<float>(band_sum);
        int fm = far_max;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            fs += __shfl_xor_sync(0xffffffffu, fs, o);
            bs += __shfl_xor_sync(0xffffffffu, bs, o);
            fm = max(fm, __shfl_xor_sync(0xffffffffu, fm, o));
        }
        if ((threadIdx.x & 31) == 0) s_cost[threadIdx.x >> 5] = make_float3(fs, bs, static_cast<float>(fm));
    }
    __syncthreads();   // the histogram and the per-warp cost sums are complete
    float far_total_cost = 0.f, band_total_cost = 0.f, far_max_cost = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
        far_total_cost += s_cost[w].x;
        band_total_cost += s_cost[w].y;
        far_max_cost = fmaxf(far_max_cost, s_cost[w].z);
    }
    // A far pair costing more than 1.25 x a CTA's mean share of the whole
    // list (all heads, `grid` CTAs) would end the launch alone: it is listed
    // as its two tiles, each an item of its own, when both hold rows.  At
    // N = 32K no pair comes near that; at N = 4K the last pair of each head
    // does (its 64 key blocks are most of the launch).
    const float all_cost = static_cast<float>(Hq) * (far_total_cost + band_total_cost);
    const int split_above = static_cast<int>(fminf(2.0e9f, all_cost * 1.25f / static_cast<float>(max(grid, 1))));
    auto split_costs = [&](int b, int pair, int cost, int& ca, int& cb) {
        ca = cost;
        cb = 0;
        if (cost <= split_above) return false;
        const int a = far_tile_cost(b, 2 * pair, fl, NT), c = far_tile_cost(b, 2 * pair + 1, fl, NT);
        if (a == 0 || c == 0) return false;
        ca = a;
        cb = c;
        return true;
    };
    if (far_max_cost > static_cast<float>(split_above)) {
        for (int u = threadIdx.x; u < U; u += blockDim.x) {
            const int cost = far_pair_cost(u / NP, u % NP, fl, NT);
            int ca, cb;
            if (!split_costs(u / NP, u % NP, cost, ca, cb)) continue;
            atomicSub(&hist[min(cost, kCostBuckets - 1)], 1);
            atomicAdd(&hist[min(ca, kCostBuckets - 1)], 1);
            atomicAdd(&hist[min(cb, kCostBuckets - 1)], 1);
        }
        __syncthreads();
    }
    // Exclusive offsets in descending cost order: thread t owns buckets
    // 4095-4t ... 4095-4t-3.
    int own = 0;
#pragma unroll
    for (int k = 0; k < kBucketsPerThread; ++k)
        own += hist[kCostBuckets - 1 - (threadIdx.x * kBucketsPerThread + k)];
    int2 totals;
    const int2 start = block_exclusive_scan2(make_int2(own, nb), warp_tot2, &totals);
    const int far_total = totals.x, band_total = totals.y;
    int run = start.x;
#pragma unroll
    for (int k = 0; k < kBucketsPerThread; ++k) {
        const int c = kCostBuckets - 1 - (threadIdx.x * kBucketsPerThread + k);
        const int h = hist[c];
        hist[c] = run;
        run += h;
    }
    __syncthreads();
    const bool coalesce = U <= kPairCache && far_total <= kPairCache;
    auto place_far = [&](int u, int kind, int cost) {
        const int pos = atomicAdd(&hist[min(cost, kCostBuckets - 1)], 1);
        if (coalesce) s_at[pos] = u | (kind << 24);
        else
            for (int h = 0; h < Hq; ++h)
                items[(size_t)h * far_total + pos] = WorkItem{kind, u / NP, h, u % NP};
    };
    for (int u = threadIdx.x; u < U; u += blockDim.x) {
        const int b = u / NP, pair = u % NP;
        const int cost = far_pair_cost(b, pair, fl, NT);
        if (cost <= 0) continue;
        int ca, cb;
        if (split_costs(b, pair, cost, ca, cb)) {
            place_far(u, kItemFarA, ca);
            place_far(u, kItemFarB, cb);
        } else {
            place_far(u, kItemFar, cost);
        }
    }
    int pos = far_total + start.y;
    for (int v = v0; v < v1; ++v) {
        int b, pair;
        band_at(v, b, pair);
        if (band_pair_cost(b, pair, tp, N, W, S, NT) <= 0) continue;
        if (coalesce) s_at[kPairCache + pos - far_total] = v;
        else
            for (int h = 0; h < Hq; ++h) items[(size_t)pos * Hq + h] = WorkItem{kItemBand, b, h, pair};
        ++pos;
    }
    if (coalesce) {
        __syncthreads();
        const int nfar = far_total * Hq, nall = (far_total + band_total) * Hq;
        for (int idx = threadIdx.x; idx < nall; idx += blockDim.x) {
            if (idx < nfar) {   // items[h * far_total + pos]
                const int e = s_at[idx % far_total], u = e & 0xFFFFFF;
                items[idx] = WorkItem{e >> 24, u / NP, idx / far_total, u % NP};
            } else {            // items[pos * Hq + h], pos >= far_total
                int b, pair;
                band_at(s_at[kPairCache + (idx - nfar) / Hq], b, pair);
                items[idx] = WorkItem{kItemBand, b, (idx - nfar) % Hq, pair};
            }
        }
    }
    if (threadIdx.x == 0) {
        n_items[0] = (far_total + band_total) * Hq;
        n_items[1] = 0;   // work counter the attention kernel claims items from
    }
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(
    const uint8_t* __restrict__ gate, int B, int N, int Hq, int W, int S, int grid,
    int* __restrict__ routed_list, int* __restrict__ routed_count, int* __restrict__ tile_prefix,
    int* __restrict__ far_last, WorkItem* __restrict__ items, int* __restrict__ n_items) {
    // The attention kernel after it is a programmatic dependent launch: let
    // its CTAs start now (they wait for this grid before reading the list).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    plan_block(gate, B, N, Hq, W, S, grid, routed_list, routed_count, tile_prefix, far_last, items,
               n_items);
}

// Router GEMV fused with the schedule: every CTA computes logits and gates of
// its tokens (each warp two tokens at a time); the CTA that finishes last (ticket from a
// counter zeroed before the launch) then plans the prefill over all gates.
// Every thread fences its gate writes before the CTA takes its ticket, and
// the last CTA fences after taking it, before reading the gates.
template <typename T>
__global__ void __launch_bounds__(kPlanThreads) route_plan_kernel(
    const uint4* __restrict__ h, const uint4* __restrict__ w, float bias, int nvec,
    float* __restrict__ logits, uint8_t* __restrict__ gate, int B, int N, int Hq, int W, int S,
    int grid, unsigned int* __restrict__ ticket, int* __restrict__ routed_list,
    int* __restrict__ routed_count, int* __restrict__ tile_prefix, int* __restrict__ far_last,
    WorkItem* __restrict__ items, int* __restrict__ n_items) {
    __shared__ int last;
    // No early trigger for the attention kernel after it: letting its CTAs
    // launch while this grid's GEMV ran made the single-layer call 4 % slower
    // (0.0871 against 0.0834 ms); it launches when this grid completes.
    const int64_t tokens = (int64_t)B * N;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    int64_t t = warp0;
    for (; t + nwarps < tokens; t += 2 * nwarps) route_token2<T>(h, w, bias, t, t + nwarps, nvec, logits, gate);
    if (t < tokens) route_token<T>(h, w, bias, t, nvec, logits, gate);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        last = atomicAdd(ticket, 1u) == gridDim.x - 1 ? 1 : 0;
        if (last) __threadfence();
    }
    __syncthreads();
    if (!last) return;
    plan_block(gate, B, N, Hq, W, S, grid, routed_list, routed_count, tile_prefix, far_last, items,
               n_items);
}

}  // namespace

PrefillWs prefill_ws_layout(int B, int N, int Hq, int d) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t NT = (static_cast<size_t>(N) + kBM - 1) / kBM;
    PrefillWs L;
    size_t off = 0;
    L.routed_list = off;
    off = up(off + sizeof(int) * (size_t)B * N);
    L.routed_count = off;
    off = up(off + sizeof(int) * (size_t)B);
    L.tile_prefix = off;
    off = up(off + sizeof(int) * (size_t)B * (NT + 1));
    L.far_last = off;
    off = up(off + sizeof(int) * (size_t)B * NT);
    L.n_items = off;
    off = up(off + sizeof(int) * 4);
    // Per batch and head at most one far pair per 256 rows, each listed whole
    // or as its two tiles, and one band pair per 256 rows.
    L.max_items = static_cast<int>((size_t)B * 3 * ((N + 2 * kBM - 1) / (2 * kBM)) * Hq);
    L.items = off;
    off = up(off + sizeof(WorkItem) * (size_t)L.max_items);
    L.total = off;
    return L;
}

cudaError_t launch_schedule(const uint8_t* gate, int B, int N, int Hq, int W, int S, int grid,
                            const PrefillWs& L, char* ws, cudaStream_t s) {
    plan_kernel<<<1, kPlanThreads, 0, s>>>(
        gate, B, N, Hq, W, S, grid, reinterpret_cast<int*>(ws + L.routed_list),
        reinterpret_cast<int*>(ws + L.routed_count), reinterpret_cast<int*>(ws + L.tile_prefix),
        reinterpret_cast<int*>(ws + L.far_last), reinterpret_cast<WorkItem*>(ws + L.items),
        reinterpret_cast<int*>(ws + L.n_items));
    return cudaGetLastError();
}

cudaError_t launch_route_plan(const void* h, const void* w, float bias, int d_model, int dtype,
                              float* logits, uint8_t* gate, int B, int N, int Hq, int W, int S,
                              const PrefillWs& L, char* ws, unsigned int* ticket, int num_sms,
                              cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(ticket, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    const int64_t tokens = (int64_t)B * N;
    const int64_t want = (tokens + kPlanThreads / 32 - 1) / (kPlanThreads / 32);
    const int blocks = static_cast<int>(want < (int64_t)num_sms ? want : (int64_t)num_sms);
    int* list = reinterpret_cast<int*>(ws + L.routed_list);
    int* count = reinterpret_cast<int*>(ws + L.routed_count);
    int* prefix = reinterpret_cast<int*>(ws + L.tile_prefix);
    int* far_last = reinterpret_cast<int*>(ws + L.far_last);
    WorkItem* items = reinterpret_cast<WorkItem*>(ws + L.items);
    int* n_items = reinterpret_cast<int*>(ws + L.n_items);
    if (dtype == 1) {
        route_plan_kernel<__nv_bfloat16><<<blocks, kPlanThreads, 0, s>>>(
            static_cast<const uint4*>(h), static_cast<const uint4*>(w), bias, d_model / 8, logits,
            gate, B, N, Hq, W, S, num_sms, ticket, list, count, prefix, far_last, items, n_items);
    } else {
        route_plan_kernel<float><<<blocks, kPlanThreads, 0, s>>>(
            static_cast<const uint4*>(h), static_cast<const uint4*>(w), bias, d_model / 4, logits,
            gate, B, N, Hq, W, S, num_sms, ticket, list, count, prefix, far_last, items, n_items);
    }
    return cudaGetLastError();
}

cudaError_t launch_far_scan(const uint8_t* gate, int B, int N, int W, int* routed_list,
                            int* routed_count, int* tile_prefix, cudaStream_t s) {
    scan_far_rows_kernel<<<B, kScanThreads, 0, s>>>(gate, N, W, routed_list, routed_count,
                                                    tile_prefix);
    return cudaGetLastError();
}

}  // namespace swi
