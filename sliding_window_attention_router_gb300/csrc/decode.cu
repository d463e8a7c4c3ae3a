// Decode over a KV cache shared by both branches (SwiAttn report, section 2:
// the two branches share the KV cache; section 6: decode reads either the
// window or the whole history).  A window token reads the last W cache
// entries, a routed one all L: the bytes moved are the whole cost.
//
// Split-KV: each chunk of `chunk` consecutive tokens of a visited range is
// streamed by one CTA (persistent CTAs claim chunks for batches of up to 32
// sequences; larger batches launch one CTA per chunk slot).  A token's K (or
// V) row for every KV head is one contiguous Hkv*d run, so each thread issues
// one 16-byte load per token and tensor, and the whole CTA reads it fully
// coalesced.  Threads of one KV head (d/VEC
// consecutive lanes) reduce q.k with xor-shuffles; each holds VEC output
// columns of the G = Hq/Hkv query heads of its group.  Partial (m, l, o) per
// chunk go to the workspace; a second kernel merges them by log-sum-exp.

#include "swiattn.h"
#include "swiattn_internal.h"

#include <cuda_bf16.h>
#include <math.h>
#include <algorithm>
#include <atomic>

namespace swi {
namespace {

constexpr int kChunk = 256;   // largest chunk (tokens per split)
constexpr int kMinChunk = 64;
constexpr int kSplit = 16;    // a visit shorter than kSplit * kChunk splits into about kSplit chunks
constexpr int kUnroll = 8;    // tokens in flight per thread

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const uint4& u, float* f) {
        const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 a = __bfloat1622float2(x[t]);
            f[2 * t] = a.x;
            f[2 * t + 1] = a.y;
        }
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const uint4& u, float* f) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
};

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Visited cache entries of sequence b: the window (or whole history)
// [lo, lo + n) and, for a window query with S global anchors, the anchors
// the window does not reach, [0, na) with na = min(S, lo).  A length outside
// [1, Lmax] is clamped into it (the split kernel reports it).  Chunks never
// straddle the two segments: the first ceil(na / chunk) chunks read anchors.
// The chunk length is about (na + n) / 16 rounded up to a power of two within
// [64, 256]: short visited ranges (windows) still split over several CTAs,
// long ones stream 256 tokens per chunk.  It depends on the sequence alone, so
// a sequence's result does not depend on the rest of the batch.
struct Visit {
    int lo, n, na, nca;   // nca: anchor chunks
    int chunk;
};
__device__ __forceinline__ int chunk_of(int m) {
    int c = kMinChunk;
    while (c < kChunk && c * kSplit < m) c <<= 1;
    return c;
}
__device__ __forceinline__ Visit visited(const int32_t* seq_lens, const uint8_t* gate, int b,
                                         int W, int S, int Lmax) {
    Visit v;
    const int L = min(max(seq_lens[b], 1), Lmax);
    const int pos = L - 1;
    v.lo = gate[b] ? 0 : max(0, pos - W + 1);
    v.n = L - v.lo;
    v.na = min(S, v.lo);
    v.chunk = chunk_of(v.na + v.n);
    v.nca = (v.na + v.chunk - 1) / v.chunk;
    return v;
}

__device__ __forceinline__ int chunks_of(const Visit& v) {
    return v.nca + (v.n + v.chunk - 1) / v.chunk;
}

// Batches up to this size dispatch their chunks longest visit first.
constexpr int kOrderMaxB = 32;

// Where token rows live: a contiguous cache [B, Lmax, Hkv, d] (Lmax rows per
// sequence), or pages [num_pages, page_size, Hkv, d] found through a block
// table [B, max_pages] (page_size = 1 << page_lg).
struct Paging {
    const int32_t* block_table;   // nullptr: contiguous
    int max_pages, page_lg, num_pages;
    unsigned int* err;
};

// NG thread groups per CTA (1 or 2) split a chunk's tokens between them, in
// alternating runs of kUnroll tokens, and merge their partials through shared
// memory at the end: twice the loads in flight per chunk where a token row
// takes at most 256 threads.
template <typename T, int D, int G, bool PAGED, int NG>
__device__ __forceinline__ void decode_split_body(const T* __restrict__ q, const T* __restrict__ kc,
                                    const T* __restrict__ vc, const int32_t* __restrict__ seq_lens,
                                    const uint8_t* __restrict__ gate, float* __restrict__ part,
                                    int Lmax, int Hq, int Hkv, int W, int S, float scale_log2,
                                    int B, int max_chunks, Paging pg, int* claim) {
    constexpr int VEC = Vec<T>::N;
    constexpr int LPH = D / VEC;   // lanes per KV head
    // For B <= 32 the CTAs are persistent: warp 0 keeps the batch's chunk
    // ranking (sequences with more chunks first, ties by index) in registers
    // and claims chunk after chunk for the CTA from the workspace counter, so
    // the longest visits start first and no CTA is launched without work.
    // Larger batches map CTA (x, y) to chunk x of sequence y, one per CTA.
    __shared__ int s_bc[2][2];
    int rk_n = 0, rk_start = 0, rk_total = 0;
    if (B <= kOrderMaxB && threadIdx.x < 32) {
        const int l = threadIdx.x;
        rk_n = l < B ? chunks_of(visited(seq_lens, gate, l, W, S, Lmax)) : 0;
        for (int o = 0; o < B; ++o) {
            const int no = __shfl_sync(0xffffffffu, rk_n, o);
            if (no > rk_n || (no == rk_n && o < l)) rk_start += no;
            rk_total += no;
        }
    }
    for (int it = 0;; ++it) {
    // Chunk of this iteration (b < 0: none).  The two slots alternate, so
    // warp 0 never overwrites a slot another warp has yet to read.
    int* bc = s_bc[it & 1];
    if (threadIdx.x < 32) {
        const int l = threadIdx.x;
        int cb = -1, cc = 0;
        if (B > kOrderMaxB) {
            if (it == 0 && (int)blockIdx.x < chunks_of(visited(seq_lens, gate, blockIdx.y, W, S, Lmax))) {
                cb = blockIdx.y;
                cc = blockIdx.x;
            }
        } else {
            int i = 0;
            if (l == 0) i = atomicAdd(claim, 1);
            i = __shfl_sync(0xffffffffu, i, 0);
            if (i < rk_total) {
                const unsigned hit = __ballot_sync(0xffffffffu, l < B && i >= rk_start && i < rk_start + rk_n);
                cb = __ffs(hit) - 1;
                cc = i - __shfl_sync(0xffffffffu, rk_start, cb);
            }
        }
        if (l == 0) {
            bc[0] = cb;
            bc[1] = cc;
        }
    }
    __syncthreads();
    const int b = bc[0], c = bc[1];
    if (b < 0) break;
    const Visit vis = visited(seq_lens, gate, b, W, S, Lmax);
    if (c == 0 && threadIdx.x == 0 && pg.err) {
        const int raw = seq_lens[b];
        if (raw < 1 || raw > Lmax) atomicOr(pg.err, kDevErrInput);
    }
    int t0, t1;   // this chunk's cache entries (the chunk is never empty)
    if (c < vis.nca) {
        t0 = c * vis.chunk;
        t1 = min(vis.na, t0 + vis.chunk);
    } else {
        t0 = vis.lo + (c - vis.nca) * vis.chunk;
        t1 = min(vis.lo + vis.n, t0 + vis.chunk);
    }
    // Paged: the physical page of every page this chunk touches, in shared
    // memory (at most kChunk + 1 of them).  An entry outside [0, num_pages)
    // is replaced by page 0 and flagged as bad input.
    __shared__ int s_page[PAGED ? kChunk + 1 : 1];
    int page_base = 0;
    if constexpr (PAGED) {
        page_base = t0 >> pg.page_lg;
        const int np = ((t1 - 1) >> pg.page_lg) - page_base + 1;
        for (int k = threadIdx.x; k < np; k += blockDim.x) {
            // A sequence longer than its table row (seq_lens past
            // max_pages * page_size) also counts as bad input.
            const bool in_row = page_base + k < pg.max_pages;
            int phys = in_row ? pg.block_table[(size_t)b * pg.max_pages + page_base + k] : -1;
            if (phys < 0 || phys >= pg.num_pages) {
                atomicOr(pg.err, kDevErrInput);
                phys = 0;
            }
            s_page[k] = phys;
        }
        __syncthreads();
    }

    // Thread group grp (tpg threads, whole warps) takes runs grp, grp + NG, ...
    // of kUnroll tokens.  Threads past Hkv*LPH in a group mirror the last KV
    // head so shuffles stay full-warp; they write nothing.
    const int tpg = blockDim.x / NG;
    const int grp = threadIdx.x / tpg, tig = threadIdx.x % tpg;
    const int active = tig < Hkv * LPH;
    const int tid = active ? tig : (Hkv - 1) * LPH + (tig % LPH);
    const int kvh = tid / LPH, sub = tid % LPH;
    const size_t row_vecs = (size_t)Hkv * LPH;   // uint4 per token row (all KV heads)

    float qf[G][VEC], acc[G][VEC], m[G], l[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int hq = kvh * G + g;
        uint4 u = *reinterpret_cast<const uint4*>(q + ((size_t)b * Hq + hq) * D + sub * VEC);
        Vec<T>::load(u, qf[g]);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            qf[g][e] *= scale_log2;
            acc[g][e] = 0.f;
        }
        m[g] = -INFINITY;
        l[g] = 0.f;
    }

    const uint4* kb = reinterpret_cast<const uint4*>(kc) + (PAGED ? 0 : (size_t)b * Lmax * row_vecs) + tid;
    const uint4* vb = reinterpret_cast<const uint4*>(vc) + (PAGED ? 0 : (size_t)b * Lmax * row_vecs) + tid;
    for (int t = t0 + grp * kUnroll; t < t1; t += NG * kUnroll) {
        uint4 ku[kUnroll], vu[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int tt = min(t + u, t1 - 1);   // clamp: duplicates are masked below
            size_t row = (size_t)tt;
            if constexpr (PAGED) {
                const int mask = (1 << pg.page_lg) - 1;
                row = ((size_t)s_page[(tt >> pg.page_lg) - page_base] << pg.page_lg) + (tt & mask);
            }
            ku[u] = ld_stream(kb + row * row_vecs);
            vu[u] = ld_stream(vb + row * row_vecs);
        }
        float s[kUnroll][G];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float kf[VEC];
            Vec<T>::load(ku[u], kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float d0 = 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) d0 = fmaf(qf[g][e], kf[e], d0);
#pragma unroll
                for (int off = LPH / 2; off > 0; off >>= 1)
                    d0 += __shfl_xor_sync(0xffffffffu, d0, off);
                s[u][g] = (t + u < t1) ? d0 : -INFINITY;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = m[g];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) mx = fmaxf(mx, s[u][g]);
            const float corr = ex2f(m[g] - mx);
            float ps = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[g][e] *= corr;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const float p = ex2f(s[u][g] - mx);
                ps += p;
                float vf[VEC];
                Vec<T>::load(vu[u], vf);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[g][e] = fmaf(p, vf[e], acc[g][e]);
            }
            l[g] = l[g] * corr + ps;
            m[g] = mx;
        }
    }

    if constexpr (NG == 2) {
        // Group 1 hands its (m, l, o) to group 0, which merges them by
        // log-sum-exp (group 0 always has a token, so its m is finite).
        extern __shared__ float s_merge[];
        constexpr int PER = G * (VEC + 2);
        float* mine = s_merge + (size_t)tig * PER;
        if (grp == 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) mine[g * (VEC + 2) + e] = acc[g][e];
                mine[g * (VEC + 2) + VEC] = m[g];
                mine[g * (VEC + 2) + VEC + 1] = l[g];
            }
        }
        __syncthreads();
        if (grp == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float m1 = mine[g * (VEC + 2) + VEC], l1 = mine[g * (VEC + 2) + VEC + 1];
                const float mx = fmaxf(m[g], m1);
                const float a0 = ex2f(m[g] - mx), a1 = ex2f(m1 - mx);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[g][e] = acc[g][e] * a0 + mine[g * (VEC + 2) + e] * a1;
                l[g] = l[g] * a0 + l1 * a1;
                m[g] = mx;
            }
        }
    }
    if (active && grp == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int hq = kvh * G + g;
            float* dst = part + (((size_t)b * max_chunks + c) * Hq + hq) * (D + 2);
#pragma unroll
            for (int e = 0; e < VEC; ++e) dst[sub * VEC + e] = acc[g][e];
            if (sub == 0) {
                dst[D] = m[g];
                dst[D + 1] = l[g];
            }
        }
    }
    }   // next chunk
    // The combine kernel is launched as a programmatic dependent of this one:
    // once every CTA has come this far it may be scheduled (it waits for this
    // grid's completion and memory before reading any partial), which hides
    // its launch behind the last CTAs' tail.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T, int D, int G, bool PAGED>
__global__ void decode_split_kernel(const T* __restrict__ q, const T* __restrict__ kc,
                                    const T* __restrict__ vc, const int32_t* __restrict__ seq_lens,
                                    const uint8_t* __restrict__ gate, float* __restrict__ part,
                                    int Lmax, int Hq, int Hkv, int W, int S, float scale_log2,
                                    int B, int max_chunks, Paging pg, int* claim) {
    decode_split_body<T, D, G, PAGED, 1>(q, kc, vc, seq_lens, gate, part, Lmax, Hq, Hkv, W, S,
                                         scale_log2, B, max_chunks, pg, claim);
}

// Two thread groups per CTA, at most 512 threads.  (Two such CTAs per SM would
// cap registers at 64, and the kernel then spills.)
template <typename T, int D, int G, bool PAGED>
__global__ void __launch_bounds__(512, 1)
decode_split2_kernel(const T* __restrict__ q, const T* __restrict__ kc,
                     const T* __restrict__ vc, const int32_t* __restrict__ seq_lens,
                     const uint8_t* __restrict__ gate, float* __restrict__ part, int Lmax, int Hq,
                     int Hkv, int W, int S, float scale_log2, int B, int max_chunks, Paging pg,
                     int* claim) {
    decode_split_body<T, D, G, PAGED, 2>(q, kc, vc, seq_lens, gate, part, Lmax, Hq, Hkv, W, S,
                                         scale_log2, B, max_chunks, pg, claim);
}

// Log-sum-exp merge of the chunk partials of one (sequence, query head):
// block (hq, b) of 1024 threads = 1024/D groups of D, thread (g, c) owns
// output column c for the chunks g, g + 1024/D, ...  The maximum over chunks
// is a block reduction; each group loads 16 of its chunks per round, so a
// routed 32K-token sequence's 128 partials arrive in one round; the groups'
// sums are then added in group order, so the result depends only on the
// sequence's own chunk count.  Launched as a programmatic dependent of the
// split kernel, it reads the visit (an input) and then waits for that grid's
// completion before touching any partial.
template <typename T, int D>
__global__ void __launch_bounds__(1024) decode_combine_kernel(const float* __restrict__ part,
                                                              const int32_t* __restrict__ seq_lens,
                                                              const uint8_t* __restrict__ gate,
                                                              T* __restrict__ o, float* __restrict__ lse,
                                                              int Hq, int W, int S, int Lmax,
                                                              int max_chunks) {
    constexpr int NG = 1024 / D;    // chunk groups
    constexpr int kRound = 16;      // chunks per group and load round
    __shared__ float red[32];
    __shared__ float s_acc[NG][D];
    __shared__ float s_l[NG];
    const int hq = blockIdx.x, b = blockIdx.y;
    const int col = threadIdx.x % D, grp = threadIdx.x / D;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    // The visit comes from the call's inputs, so it is read before waiting.
    const Visit vis = visited(seq_lens, gate, b, W, S, Lmax);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int nc = vis.nca + (vis.n + vis.chunk - 1) / vis.chunk;
    const float* base = part + ((size_t)b * max_chunks * Hq + hq) * (D + 2);
    const size_t cstride = (size_t)Hq * (D + 2);
    float M = -INFINITY;
    for (int c = threadIdx.x; c < nc; c += 1024) M = fmaxf(M, base[c * cstride + D]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0) red[wid] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < 32; ++w) M = fmaxf(M, red[w]);
    // Group g sums chunks g, g + NG, ...; the groups are then added in order.
    float L = 0.f, acc = 0.f;
    for (int c0 = grp; c0 < nc; c0 += NG * kRound) {
        float mv[kRound], lv[kRound], ov[kRound];
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
            const int c = c0 + u * NG;
            const float* pc = base + (size_t)(c < nc ? c : 0) * cstride;
            mv[u] = c < nc ? pc[D] : -INFINITY;
            lv[u] = c < nc ? pc[D + 1] : 0.f;
            ov[u] = c < nc ? pc[col] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kRound; ++u) {
            const float w = ex2f(mv[u] - M);
            L = fmaf(lv[u], w, L);
            acc = fmaf(ov[u], w, acc);
        }
    }
    s_acc[grp][col] = acc;
    if (col == 0) s_l[grp] = L;
    __syncthreads();
    if (grp != 0) return;
    float A = s_acc[0][col], Lt = s_l[0];
#pragma unroll
    for (int g = 1; g < NG; ++g) {
        A += s_acc[g][col];
        Lt += s_l[g];
    }
    const float val = A / Lt;
    T* dst = o + ((size_t)b * Hq + hq) * D + col;
    if constexpr (sizeof(T) == 2) {
        *dst = __float2bfloat16_rn(val);
    } else {
        *dst = val;
    }
    if (lse && col == 0) lse[(size_t)b * Hq + hq] = (M + __log2f(Lt)) * 0.69314718055994531f;
}

// Thread groups per CTA for a token row of tpg threads and G query heads per
// KV head: two groups when the row takes at most 256 threads and G <= 2 (the
// merge buffer is then at most 20 KiB), else one.  It depends on the shapes
// alone, so a sequence's result does not depend on the rest of the batch.
inline int split_groups(int tpg, int G) { return (tpg <= 256 && G <= 2) ? 2 : 1; }

inline int num_sms_of_current_device() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

// B <= 32: as many persistent CTAs as fit on the GPU at once (at most one per
// chunk slot), after clearing the claim counter on the stream; larger
// batches: one CTA per (chunk, sequence) slot.
template <typename T, int D, int G, int NG>
cudaError_t launch_split_ng(const void* q, const void* kc, const void* vc, const int32_t* sl,
                            const uint8_t* gate, float* part, int* claim, int B, int Lmax, int Hq,
                            int Hkv, int W, int S, float scale_log2, int max_chunks,
                            const Paging& pg, int tpg, cudaStream_t s) {
    const size_t smem = NG > 1 ? sizeof(float) * tpg * G * (Vec<T>::N + 2) : 0;
    using Kern = void (*)(const T*, const T*, const T*, const int32_t*, const uint8_t*, float*,
                          int, int, int, int, int, float, int, int, Paging, int*);
    Kern kern;
    if constexpr (NG == 2)
        kern = pg.block_table ? decode_split2_kernel<T, D, G, true> : decode_split2_kernel<T, D, G, false>;
    else
        kern = pg.block_table ? decode_split_kernel<T, D, G, true> : decode_split_kernel<T, D, G, false>;
    dim3 grid(max_chunks, B);
    if (B <= kOrderMaxB) {
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NG * tpg, smem);
        if (e != cudaSuccess) return e;
        const int sms = num_sms_of_current_device();
        if (sms <= 0) return cudaErrorInvalidDevice;
        const int64_t slots = (int64_t)max_chunks * B;
        grid = dim3((unsigned)std::min<int64_t>(slots, (int64_t)sms * std::max(per_sm, 1)));
        e = cudaMemsetAsync(claim, 0, sizeof(int), s);
        if (e != cudaSuccess) return e;
    }
    kern<<<grid, NG * tpg, smem, s>>>(static_cast<const T*>(q), static_cast<const T*>(kc),
                                      static_cast<const T*>(vc), sl, gate, part, Lmax, Hq, Hkv, W,
                                      S, scale_log2, B, max_chunks, pg, claim);
    return cudaGetLastError();
}

template <typename T, int D, int G>
cudaError_t launch_split(const void* q, const void* kc, const void* vc, const int32_t* sl,
                         const uint8_t* gate, float* part, int* claim, int B, int Lmax, int Hq,
                         int Hkv, int W, int S, float scale_log2, int max_chunks, const Paging& pg,
                         cudaStream_t s) {
    const int tpg = (Hkv * (D / Vec<T>::N) + 31) / 32 * 32;
    if constexpr (G <= 2) {
        if (split_groups(tpg, G) == 2)
            return launch_split_ng<T, D, G, 2>(q, kc, vc, sl, gate, part, claim, B, Lmax, Hq, Hkv,
                                               W, S, scale_log2, max_chunks, pg, tpg, s);
    }
    return launch_split_ng<T, D, G, 1>(q, kc, vc, sl, gate, part, claim, B, Lmax, Hq, Hkv, W, S,
                                       scale_log2, max_chunks, pg, tpg, s);
}

template <typename T, int D>
cudaError_t launch_typed(const void* q, const void* kc, const void* vc, const int32_t* sl,
                         const uint8_t* gate, void* o, float* lse, int B, int Lmax, int Hq,
                         int Hkv, int W, int S, float scale, float* part, int* claim,
                         int max_chunks, const Paging& pg, cudaStream_t s) {
    const float sl2 = scale * 1.4426950408889634f;
    const int G = Hq / Hkv;
    cudaError_t e;
    prof_start(s);
    switch (G) {
        case 1: e = launch_split<T, D, 1>(q, kc, vc, sl, gate, part, claim, B, Lmax, Hq, Hkv, W, S, sl2, max_chunks, pg, s); break;
        case 2: e = launch_split<T, D, 2>(q, kc, vc, sl, gate, part, claim, B, Lmax, Hq, Hkv, W, S, sl2, max_chunks, pg, s); break;
        case 4: e = launch_split<T, D, 4>(q, kc, vc, sl, gate, part, claim, B, Lmax, Hq, Hkv, W, S, sl2, max_chunks, pg, s); break;
        case 8: e = launch_split<T, D, 8>(q, kc, vc, sl, gate, part, claim, B, Lmax, Hq, Hkv, W, S, sl2, max_chunks, pg, s); break;
        default: return cudaErrorInvalidValue;
    }
    prof_stop(s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(Hq, B);
    cfg.blockDim = dim3(1024);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<T, D>, static_cast<const float*>(part), sl,
                           gate, static_cast<T*>(o), lse, Hq, W, S, Lmax, max_chunks);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_decode_any(const void* q, const void* kc, const void* vc,
                              const int32_t* seq_lens, const uint8_t* gate, void* o, float* lse,
                              int B, int Lmax, int Hq, int Hkv, int d, int W, int S,
                              float scale, int dtype, const DecodeWs& L, char* ws,
                              const Paging& pg, cudaStream_t s) {
    float* part = reinterpret_cast<float*>(ws + L.part);
    int* claim = reinterpret_cast<int*>(ws + L.claim);
    if (dtype == 1) {
        if (d == 128) return launch_typed<__nv_bfloat16, 128>(q, kc, vc, seq_lens, gate, o, lse, B, Lmax, Hq, Hkv, W, S, scale, part, claim, L.max_chunks, pg, s);
        if (d == 64) return launch_typed<__nv_bfloat16, 64>(q, kc, vc, seq_lens, gate, o, lse, B, Lmax, Hq, Hkv, W, S, scale, part, claim, L.max_chunks, pg, s);
    } else {
        if (d == 128) return launch_typed<float, 128>(q, kc, vc, seq_lens, gate, o, lse, B, Lmax, Hq, Hkv, W, S, scale, part, claim, L.max_chunks, pg, s);
        if (d == 64) return launch_typed<float, 64>(q, kc, vc, seq_lens, gate, o, lse, B, Lmax, Hq, Hkv, W, S, scale, part, claim, L.max_chunks, pg, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

DecodeWs decode_ws_layout(int B, int Lmax, int Hq, int d, int S) {
    DecodeWs L;
    L.chunk = kChunk;
    // A visit of m = na + n <= Lmax + min(S, Lmax) entries has at most
    // ceil(m / chunk) + 1 chunks (ceil(a/c) + ceil(b/c) <= ceil((a+b)/c) + 1
    // for its two segments): kSplit + 1 while the chunk is below 256 (then
    // chunk * kSplit >= m), else ceil(m / 256) + 1.
    const int64_t m = (int64_t)Lmax + (S < Lmax ? S : Lmax);
    const int64_t longest = (m + kChunk - 1) / kChunk + 1;
    L.max_chunks = longest > kSplit + 1 ? (int)longest : kSplit + 1;
    L.part = 0;
    L.claim = sizeof(float) * (size_t)B * L.max_chunks * Hq * (d + 2);
    L.claim = (L.claim + 255) & ~static_cast<size_t>(255);
    L.total = L.claim + 256;
    return L;
}

cudaError_t launch_decode(const void* q, const void* kc, const void* vc, const int32_t* seq_lens,
                          const uint8_t* gate, void* o, float* lse, int B, int Lmax, int Hq,
                          int Hkv, int d, int W, int S, float scale, int dtype,
                          const DecodeWs& L, char* ws, unsigned int* err, cudaStream_t s) {
    Paging pg{nullptr, 0, 0, 0, err};
    return launch_decode_any(q, kc, vc, seq_lens, gate, o, lse, B, Lmax, Hq, Hkv, d, W, S, scale,
                             dtype, L, ws, pg, s);
}

cudaError_t launch_decode_paged(const void* q, const void* kp, const void* vp,
                                const int32_t* block_table, const int32_t* seq_lens,
                                const uint8_t* gate, void* o, float* lse, int B, int max_pages,
                                int page_lg, int num_pages, int Hq, int Hkv, int d, int W, int S,
                                float scale, int dtype, const DecodeWs& L, char* ws,
                                unsigned int* err, cudaStream_t s) {
    Paging pg{block_table, max_pages, page_lg, num_pages, err};
    return launch_decode_any(q, kp, vp, seq_lens, gate, o, lse, B, max_pages << page_lg, Hq, Hkv,
                             d, W, S, scale, dtype, L, ws, pg, s);
}

namespace {

// Largest block the split kernel can launch with: its register use bounds it
// below 1024 threads (read from the compiled kernel, cached per kind).
template <typename T, int D, int G>
int split_block_cap(bool paged) {
    static std::atomic<int> cap[2];
    int c = cap[paged].load(std::memory_order_relaxed);
    if (c > 0) return c;
    cudaFuncAttributes attr;
    const cudaError_t e = paged ? cudaFuncGetAttributes(&attr, decode_split_kernel<T, D, G, true>)
                                : cudaFuncGetAttributes(&attr, decode_split_kernel<T, D, G, false>);
    if (e != cudaSuccess) return 0;
    c = attr.maxThreadsPerBlock;
    cap[paged].store(c, std::memory_order_relaxed);
    return c;
}

template <typename T, int D>
int split_block_cap(int G, bool paged) {
    switch (G) {
        case 1: return split_block_cap<T, D, 1>(paged);
        case 2: return split_block_cap<T, D, 2>(paged);
        case 4: return split_block_cap<T, D, 4>(paged);
        case 8: return split_block_cap<T, D, 8>(paged);
        default: return 0;
    }
}

}  // namespace

int decode_block_check(int dtype, int d, int Hq, int Hkv, bool paged) {
    const int G = Hq / Hkv;
    int cap = 0;
    if (dtype == SWIATTN_BF16)
        cap = d == 128 ? split_block_cap<__nv_bfloat16, 128>(G, paged)
                       : split_block_cap<__nv_bfloat16, 64>(G, paged);
    else
        cap = d == 128 ? split_block_cap<float, 128>(G, paged) : split_block_cap<float, 64>(G, paged);
    if (cap <= 0) return SWIATTN_OK;   // limit unknown: the launch itself decides
    const int vec = dtype == SWIATTN_BF16 ? 8 : 4;
    const int64_t threads = ((int64_t)Hkv * d / vec + 31) / 32 * 32;
    return threads <= cap ? SWIATTN_OK : SWIATTN_EUNSUPPORTED;
}

}  // namespace swi
