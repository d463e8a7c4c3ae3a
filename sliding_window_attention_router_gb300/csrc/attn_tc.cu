// Dual-branch training forward on the 5th-generation tensor cores (sm_103a).
//
// One persistent CTA per SM walks the 128-row query tiles of every
// (batch, head), latest (longest) tiles first.  Per tile it
// streams 128-key K/V blocks with TMA into 128-byte-swizzled shared memory,
// computes S = Q K^T with tcgen05.mma into TMEM, runs an fp32 online softmax
// (one thread per query row, exp2 on the MUFU), writes P as bf16 back to
// shared memory and accumulates O += P V in TMEM.  Warp roles:
//   warps 0-3  softmax + epilogue (thread r owns query row r == TMEM lane r)
//   warp 4     TMA producer for Q and K
//   warp 5     TMEM allocator and single-thread MMA issuer
//   warp 6     TMA producer for V
// All hand-offs are shared-memory mbarriers with bounded waits.
//
// Per tile (SwiAttn report, section 2, dual-branch computation; window per the
// weimeta.cn SWA glossary, "详细解释"): the window keys [max(0, i-W+1), i]
// first, then O/l is snapshotted as O_SWA (kept in TMEM, written as bf16),
// then the remaining keys [0, i-W] complete O_FULL.  The epilogue writes
// O_FULL, the gated output and each row's squared distance ||o_FULL - o_SWA||^2
// for its head, from the fp32 values.

#include "ptx.cuh"
#include "swiattn_internal.h"

#include <cuda_bf16.h>
#include <math.h>

namespace swi {
namespace {

constexpr int kStages = 2;
constexpr int kThreads = 224;
constexpr int kTileBytes = kBM * kHD * 2;    // 32 KiB: 128 rows x 128 bf16
constexpr int kHalfBytes = kTileBytes / 2;   // 16 KiB: 128 rows x 64 bf16 (one swizzle column)

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffP = kOffV + kStages * kTileBytes;
constexpr int kOffBar = kOffP + kTileBytes;

enum {
    BAR_Q_FULL = 0,
    BAR_Q_EMPTY,
    BAR_K_FULL,
    BAR_K_EMPTY = BAR_K_FULL + kStages,
    BAR_V_FULL = BAR_K_EMPTY + kStages,
    BAR_V_EMPTY = BAR_V_FULL + kStages,
    BAR_S_FULL = BAR_V_EMPTY + kStages,
    BAR_S_EMPTY = BAR_S_FULL + 2,
    BAR_P_FULL = BAR_S_EMPTY + 2,
    BAR_PV_DONE,
    BAR_O_FREE,
    BAR_DRAIN,
    BAR_COUNT
};

constexpr int kOffMisc = kOffBar + BAR_COUNT * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;   // + TMEM address, abort flag, alignment slack

constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColSnap = 384, kTmemCols = 512;

constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);   // Q: K-major, K: K-major
constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, kHD, false, true);    // P: K-major, V: MN-major

struct TcParams {
    CUtensorMap tm_q;    // Q  [B,N,Hq,128], box 64 x 1 x 128 x 1
    CUtensorMap tm_k;    // K  [B,N,Hkv,128]
    CUtensorMap tm_v;    // V
    const float* logits;
    __nv_bfloat16* o;        // O_FULL
    __nv_bfloat16* o_swa;
    __nv_bfloat16* o_gated;  // nullable
    float* mse_part;         // [B,N,Hq] squared distance per (token, head)
    unsigned int* err;
    int B, N, Hq, Hkv, W;
    float scale_log2;
};

// What one work item asks for.
struct Plan {
    int b, h, kvh;
    int row0, nrows;   // first query row, valid rows
    int kv1, nblk1;    // window keys: first key and block count
    int kv2, nblk2;    // remaining keys [0, i-W]
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int item_count(const TcParams& p) { return p.B * p.Hq * cdiv(p.N, kBM); }

// Snake order over the cost-ordered items: CTA c takes items c, 2G-1-c,
// 2G+c, 4G-1-c, ... so every CTA gets one item of every rank band.
__device__ __forceinline__ int snake_index(int k, int c, int G) {
    return k * G + ((k & 1) ? (G - 1 - c) : c);
}

__device__ __forceinline__ Plan make_plan(const TcParams& p, int idx) {
    Plan pl;
    const int nqt = cdiv(p.N, kBM);
    const int per = p.B * p.Hq;
    const int tile = nqt - 1 - idx / per;   // longest (latest) tiles first
    const int rem = idx % per;
    pl.b = rem / p.Hq;
    pl.h = rem % p.Hq;
    pl.kvh = pl.h / (p.Hq / p.Hkv);
    pl.row0 = tile * kBM;
    pl.nrows = min(kBM, p.N - pl.row0);
    const int hi_row = pl.row0 + pl.nrows - 1;
    pl.kv1 = max(0, pl.row0 - p.W + 1);
    pl.nblk1 = cdiv(hi_row - pl.kv1 + 1, kBN);
    pl.kv2 = 0;
    const int far_hi = hi_row - p.W;
    pl.nblk2 = far_hi >= 0 ? cdiv(far_hi + 1, kBN) : 0;
    return pl;
}

__device__ __forceinline__ int block_key0(const Plan& pl, int j) {
    return j < pl.nblk1 ? pl.kv1 + j * kBN : pl.kv2 + (j - pl.nblk1) * kBN;
}

// ----------------------------------------------------------------- roles --

__device__ bool producer_qk(const TcParams& p, uint8_t* smem, uint64_t* bar, volatile int* abort_flag,
                            uint32_t& kv_issued, uint32_t& q_issued) {
    const int G = gridDim.x, c = blockIdx.x;
    const int n = item_count(p);
    for (int k = 0;; ++k) {
        const int idx = snake_index(k, c, G);
        if (idx >= n) break;
        const Plan pl = make_plan(p, idx);
        if (!mbar_wait(&bar[BAR_Q_EMPTY], (q_issued & 1u) ^ 1u, abort_flag, p.err)) return false;
        mbar_arrive_expect_tx(&bar[BAR_Q_FULL], kTileBytes);
        tma_load_4d(smem + kOffQ, &p.tm_q, &bar[BAR_Q_FULL], 0, pl.h, pl.row0, pl.b);
        tma_load_4d(smem + kOffQ + kHalfBytes, &p.tm_q, &bar[BAR_Q_FULL], 64, pl.h, pl.row0, pl.b);
        ++q_issued;
        const int nblk = pl.nblk1 + pl.nblk2;
        for (int j = 0; j < nblk; ++j) {
            const uint32_t st = kv_issued % kStages, ph = (kv_issued / kStages) & 1u;
            if (!mbar_wait(&bar[BAR_K_EMPTY + st], ph ^ 1u, abort_flag, p.err)) return false;
            mbar_arrive_expect_tx(&bar[BAR_K_FULL + st], kTileBytes);
            uint8_t* dst = smem + kOffK + st * kTileBytes;
            const int key0 = block_key0(pl, j);
            tma_load_4d(dst, &p.tm_k, &bar[BAR_K_FULL + st], 0, pl.kvh, key0, pl.b);
            tma_load_4d(dst + kHalfBytes, &p.tm_k, &bar[BAR_K_FULL + st], 64, pl.kvh, key0, pl.b);
            ++kv_issued;
        }
    }
    return true;
}

__device__ bool producer_v(const TcParams& p, uint8_t* smem, uint64_t* bar, volatile int* abort_flag,
                           uint32_t& kv_issued) {
    const int G = gridDim.x, c = blockIdx.x;
    const int n = item_count(p);
    for (int k = 0;; ++k) {
        const int idx = snake_index(k, c, G);
        if (idx >= n) break;
        const Plan pl = make_plan(p, idx);
        const int nblk = pl.nblk1 + pl.nblk2;
        for (int j = 0; j < nblk; ++j) {
            const uint32_t st = kv_issued % kStages, ph = (kv_issued / kStages) & 1u;
            if (!mbar_wait(&bar[BAR_V_EMPTY + st], ph ^ 1u, abort_flag, p.err)) return false;
            mbar_arrive_expect_tx(&bar[BAR_V_FULL + st], kTileBytes);
            uint8_t* dst = smem + kOffV + st * kTileBytes;
            const int key0 = block_key0(pl, j);
            tma_load_4d(dst, &p.tm_v, &bar[BAR_V_FULL + st], 0, pl.kvh, key0, pl.b);
            tma_load_4d(dst + kHalfBytes, &p.tm_v, &bar[BAR_V_FULL + st], 64, pl.kvh, key0, pl.b);
            ++kv_issued;
        }
    }
    return true;
}

// After an abort: wait (briefly, bounded) for TMA copies this thread issued
// that nobody consumed, so no copy lands in shared memory after exit.
__device__ void drain_loads(uint64_t* full_bars, uint32_t issued) {
    for (uint32_t back = 1; back <= kStages && back <= issued; ++back) {
        const uint32_t it = issued - back;
        mbar_drain(&full_bars[it % kStages], (it / kStages) & 1u);
    }
}

__device__ bool mma_issuer(const TcParams& p, uint8_t* smem, uint64_t* bar, uint32_t tmem,
                           volatile int* abort_flag) {
    const int G = gridDim.x, c = blockIdx.x;
    const int n = item_count(p);
    const uint32_t sQ = smem_u32(smem + kOffQ);
    const uint32_t sP = smem_u32(smem + kOffP);
    uint32_t kv_iter = 0, s_iter = 0, pv_iter = 0, q_iter = 0, o_iter = 0;

    auto issue_pv = [&](uint32_t kv_index, bool first) -> bool {
        const uint32_t st = kv_index % kStages, ph = (kv_index / kStages) & 1u;
        if (!mbar_wait(&bar[BAR_P_FULL], pv_iter & 1u, abort_flag, p.err)) return false;
        if (!mbar_wait(&bar[BAR_V_FULL + st], ph, abort_flag, p.err)) return false;
        if (first) {
            if (!mbar_wait(&bar[BAR_O_FREE], (o_iter & 1u) ^ 1u, abort_flag, p.err)) return false;
            ++o_iter;
        }
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + kOffV + st * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t a = sdesc_sw128(sP + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t bdesc = sdesc_sw128(sV + kk * 16 * 128, kHalfBytes, 1024);
            umma_bf16(tmem + kColO, a, bdesc, kIdescO, (first && kk == 0) ? 0u : 1u);
        }
        umma_commit(&bar[BAR_PV_DONE]);
        umma_commit(&bar[BAR_V_EMPTY + st]);
        ++pv_iter;
        return true;
    };

    for (int k = 0;; ++k) {
        const int idx = snake_index(k, c, G);
        if (idx >= n) break;
        const Plan pl = make_plan(p, idx);
        if (!mbar_wait(&bar[BAR_Q_FULL], q_iter & 1u, abort_flag, p.err)) return false;
        ++q_iter;
        tc_fence_after();
        const int nblk = pl.nblk1 + pl.nblk2;
        for (int j = 0; j < nblk; ++j) {
            const uint32_t kvi = kv_iter + j;
            const uint32_t st = kvi % kStages, ph = (kvi / kStages) & 1u;
            const uint32_t sb = s_iter & 1u;
            if (!mbar_wait(&bar[BAR_K_FULL + st], ph, abort_flag, p.err)) return false;
            if (!mbar_wait(&bar[BAR_S_EMPTY + sb], ((s_iter >> 1) & 1u) ^ 1u, abort_flag, p.err))
                return false;
            tc_fence_after();
            const uint32_t sK = smem_u32(smem + kOffK + st * kTileBytes);
            const uint32_t dS = tmem + (sb ? kColS1 : kColS0);
#pragma unroll
            for (int kk = 0; kk < kHD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                umma_bf16(dS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024),
                          kIdescS, kk > 0 ? 1u : 0u);
            }
            umma_commit(&bar[BAR_S_FULL + sb]);
            umma_commit(&bar[BAR_K_EMPTY + st]);
            if (j == nblk - 1) umma_commit(&bar[BAR_Q_EMPTY]);
            ++s_iter;
            if (j >= 1 && !issue_pv(kvi - 1, j == 1)) return false;
        }
        if (!issue_pv(kv_iter + nblk - 1, nblk == 1)) return false;
        kv_iter += nblk;
    }
    return true;
}

// Per-row key range of block j for the softmax role; empty when i < 0.
__device__ __forceinline__ void row_range(const Plan& pl, int j, int i, int W, int& lo, int& hi) {
    if (i < 0) {
        lo = 1;
        hi = 0;
    } else if (j >= pl.nblk1) {   // keys beyond the window
        lo = 0;
        hi = i - W;
    } else {
        lo = max(0, i - W + 1);
        hi = i;
    }
}

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float* v, int n32) {
    // n32 consecutive groups of 8 values -> 16-byte stores
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int g = 0; g < n32; ++g) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * g + 0], v[8 * g + 1]);
        w.y = pack_bf16x2(v[8 * g + 2], v[8 * g + 3]);
        w.z = pack_bf16x2(v[8 * g + 4], v[8 * g + 5]);
        w.w = pack_bf16x2(v[8 * g + 6], v[8 * g + 7]);
        d4[g] = w;
    }
}

// Softmax warps run warp-collective TMEM instructions after their waits, so
// a wait only counts as passed when it passed for every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err) {
    const bool ok = mbar_wait(bar, parity, abort_flag, err);
    return __all_sync(0xffffffffu, ok);
}

__device__ bool softmax_role(const TcParams& p, uint8_t* smem, uint64_t* bar, uint32_t tmem,
                             volatile int* abort_flag, int warp, int lane) {
    const int G = gridDim.x, c = blockIdx.x;
    const int n = item_count(p);
    const int r = warp * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t sP = smem_u32(smem + kOffP);
    const float sl = p.scale_log2;
    uint32_t s_iter = 0, pv_iter = 0;

    for (int k = 0;; ++k) {
        const int idx = snake_index(k, c, G);
        if (idx >= n) break;
        const Plan pl = make_plan(p, idx);
        const int i = (r < pl.nrows) ? pl.row0 + r : -1;
        const size_t out_row = (i >= 0) ? (((size_t)pl.b * p.N + i) * p.Hq + pl.h) : 0;

        float m2 = -INFINITY, l = 0.f;
        bool snapped = false;
        const int nblk = pl.nblk1 + pl.nblk2;
        for (int j = 0; j < nblk; ++j) {
            int lo, hi;
            row_range(pl, j, i, p.W, lo, hi);
            const int key0 = block_key0(pl, j);
            const int a = lo - key0, e = hi - key0;   // valid columns [a, e]
            const uint32_t sb = s_iter & 1u;
            if (!warp_wait(&bar[BAR_S_FULL + sb], (s_iter >> 1) & 1u, abort_flag, p.err)) return false;
            tc_fence_after();
            uint32_t sr[128];
            const uint32_t tS = lane_base + (sb ? kColS1 : kColS0);
            tmem_ld32(tS + 0, sr);
            tmem_ld32(tS + 32, sr + 32);
            tmem_ld32(tS + 64, sr + 64);
            tmem_ld32(tS + 96, sr + 96);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bar[BAR_S_EMPTY + sb]);
            ++s_iter;

            float* s = reinterpret_cast<float*>(sr);
            // Eight independent partial maxima keep the dependency chains short.
            float m8[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) m8[t] = -INFINITY;
            if (a <= 0 && e >= kBN - 1) {
#pragma unroll
                for (int cc = 0; cc < kBN; ++cc) m8[cc & 7] = fmaxf(m8[cc & 7], s[cc]);
            } else {
#pragma unroll
                for (int cc = 0; cc < kBN; ++cc) {
                    s[cc] = (cc >= a && cc <= e) ? s[cc] : -INFINITY;
                    m8[cc & 7] = fmaxf(m8[cc & 7], s[cc]);
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            // Running max in scaled log2 units; O and l are only rescaled when
            // the max grows by more than 2^8, otherwise p stays <= 256.
            const float mnew = fmaxf(m2, mx * sl);
            const bool resc = mnew > m2 + 8.0f;
            float alpha = 1.f;
            if (resc) {
                alpha = ex2_approx(m2 - mnew);
                m2 = mnew;
            }
            const float mb = (m2 == -INFINITY) ? 0.f : m2;
            float r8[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) r8[t] = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int cc = 0; cc < kBN; cc += 2) {
                const float p0 = ex2_approx(fmaf(s[cc], sl, -mb));
                const float p1 = ex2_approx(fmaf(s[cc + 1], sl, -mb));
                r8[(cc >> 1) & 7] += p0 + p1;
                pk[cc >> 1] = pack_bf16x2(p0, p1);
            }
            const float rs = ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));

            if (j >= 1) {
                // P buffer free and O stable once the previous PV completed.
                if (!warp_wait(&bar[BAR_PV_DONE], pv_iter & 1u, abort_flag, p.err)) return false;
                ++pv_iter;
                tc_fence_after();
                if (j == pl.nblk1) {
                    // End of the window keys: O/l is this row's O_SWA.
                    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t orr[32];
                        tmem_ld32(lane_base + kColO + q4 * 32, orr);
                        tmem_ld_wait();
                        float* ov = reinterpret_cast<float*>(orr);
#pragma unroll
                        for (int t = 0; t < 32; ++t) ov[t] *= inv;
                        tmem_st32(lane_base + kColSnap + q4 * 32, orr);
                        if (i >= 0) store_row_bf16(p.o_swa + out_row * kHD + q4 * 32, ov, 4);
                    }
                    tmem_st_wait();
                    snapped = true;
                }
                const bool need = resc && l > 0.f;
                if (__any_sync(0xffffffffu, need)) {
                    const float f = need ? alpha : 1.f;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t orr[32];
                        tmem_ld32(lane_base + kColO + q4 * 32, orr);
                        tmem_ld_wait();
                        float* ov = reinterpret_cast<float*>(orr);
#pragma unroll
                        for (int t = 0; t < 32; ++t) ov[t] *= f;
                        tmem_st32(lane_base + kColO + q4 * 32, orr);
                    }
                    tmem_st_wait();
                }
            }
            l = l * alpha + rs;

            // P row -> shared memory, K-major with the 128-byte swizzle.
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const uint32_t addr = sP + (u >> 3) * kHalfBytes + r * 128 +
                                      ((((uint32_t)u & 7u) ^ ((uint32_t)r & 7u)) << 4);
                st_shared_v4(addr, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar[BAR_P_FULL]);
        }

        // Epilogue: wait for the last PV, normalise, store.
        if (!warp_wait(&bar[BAR_PV_DONE], pv_iter & 1u, abort_flag, p.err)) return false;
        ++pv_iter;
        tc_fence_after();
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        float mse = 0.f;
        const bool gated_full = (i >= 0) ? (p.logits[(size_t)pl.b * p.N + i] > 0.f) : false;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t orr[32];
            tmem_ld32(lane_base + kColO + q4 * 32, orr);
            tmem_ld_wait();
            float* ov = reinterpret_cast<float*>(orr);
#pragma unroll
            for (int t = 0; t < 32; ++t) ov[t] *= inv;
            {
                uint32_t srr[32];
                float* sv = reinterpret_cast<float*>(srr);
                if (snapped) {
                    tmem_ld32(lane_base + kColSnap + q4 * 32, srr);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) sv[t] = ov[t];
                }
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const float dlt = ov[t] - sv[t];
                    mse = fmaf(dlt, dlt, mse);
                }
                if (i >= 0) {
                    store_row_bf16(p.o + out_row * kHD + q4 * 32, ov, 4);
                    if (!snapped) store_row_bf16(p.o_swa + out_row * kHD + q4 * 32, ov, 4);
                    if (p.o_gated) {
                        float gv[32];
#pragma unroll
                        for (int t = 0; t < 32; ++t) gv[t] = gated_full ? ov[t] : sv[t];
                        store_row_bf16(p.o_gated + out_row * kHD + q4 * 32, gv, 4);
                    }
                }
            }
        }
        if (i >= 0) p.mse_part[out_row] = mse;
        tc_fence_before();
        mbar_arrive(&bar[BAR_O_FREE]);
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) tc_attention_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bar[BAR_Q_FULL], 1);
        mbar_init(&bar[BAR_Q_EMPTY], 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar[BAR_K_FULL + s], 1);
            mbar_init(&bar[BAR_K_EMPTY + s], 1);
            mbar_init(&bar[BAR_V_FULL + s], 1);
            mbar_init(&bar[BAR_V_EMPTY + s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar[BAR_S_FULL + s], 1);
            mbar_init(&bar[BAR_S_EMPTY + s], kBM);
        }
        mbar_init(&bar[BAR_P_FULL], kBM);
        mbar_init(&bar[BAR_PV_DONE], 1);
        mbar_init(&bar[BAR_O_FREE], kBM);
        mbar_init(&bar[BAR_DRAIN], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        softmax_role(p, smem, bar, tmem, abort_flag, warp, lane);
    } else if (warp == 4) {
        if (lane == 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_k);
            uint32_t kv_issued = 0, q_issued = 0;
            if (!producer_qk(p, smem, bar, abort_flag, kv_issued, q_issued)) {
                drain_loads(&bar[BAR_K_FULL], kv_issued);
                if (q_issued) mbar_drain(&bar[BAR_Q_FULL], (q_issued - 1) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            mma_issuer(p, smem, bar, tmem, abort_flag);
            // Every MMA this thread issued has completed once this arrives.
            umma_commit(&bar[BAR_DRAIN]);
            mbar_drain(&bar[BAR_DRAIN], 0);
        }
        __syncwarp();
    } else {
        if (lane == 0) {
            prefetch_tensormap(&p.tm_v);
            uint32_t kv_issued = 0;
            if (!producer_v(p, smem, bar, abort_flag, kv_issued)) drain_loads(&bar[BAR_V_FULL], kv_issued);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_tc_attention(const TcAttnArgs& a, unsigned int* err, int num_sms,
                                cudaStream_t s) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    const uint64_t N = a.N, B = a.B;
    bool ok = make_tmap_4d_bf16(&p.tm_q, a.q, kHD, a.Hq, N, B, 64, kBM) &&
              make_tmap_4d_bf16(&p.tm_k, a.k, kHD, a.Hkv, N, B, 64, kBN) &&
              make_tmap_4d_bf16(&p.tm_v, a.v, kHD, a.Hkv, N, B, 64, kBN);
    if (!ok) return cudaErrorInvalidValue;
    p.logits = a.logits;
    p.o = static_cast<__nv_bfloat16*>(a.o);
    p.o_swa = static_cast<__nv_bfloat16*>(a.o_swa);
    p.o_gated = static_cast<__nv_bfloat16*>(a.o_gated);
    p.mse_part = a.mse_part;
    p.err = err;
    p.B = a.B;
    p.N = a.N;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.W = a.W;
    p.scale_log2 = a.scale * 1.4426950408889634f;

    static bool attr_set = false;   // per process; the attribute is per function
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_attention_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    tc_attention_kernel<<<num_sms, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace swi
