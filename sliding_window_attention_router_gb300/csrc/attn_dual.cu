// Dual-branch training forward on the 5th-generation tensor cores (sm_103a):
// both branches for every row, two query tiles per CTA sharing each K/V block.
//
// SwiAttn report, section 2 (dual-branch computation; window per the
// weimeta.cn SWA glossary, "详细解释"): each row i needs O_SWA over keys
// [max(0, i-W+1), i] and O_FULL over [0, i].  The window keys are a suffix of
// the full range, so one online softmax per row serves both: it first walks
// the window keys, then O/l is this row's O_SWA (snapshotted), then it walks
// the remaining keys [0, i-W] and O/l is O_FULL.  Every (row, key) pair is
// visited once.
//
// A work item is 256 rows of one (batch, head): tiles A (rows q0 ..) and B
// (q0+128 ..).  Its block sequence is the window sweep (128-key blocks from
// max(0, q0-W+1); tile B's run is tile A's shifted by one block) followed by
// the far sweep (blocks from key 0; each tile's run ends at its last row - W).
// Structure as in the routed prefill: P over S in TMEM, PV with A from TMEM,
// the two tiles' chains interleaved on the tensor core, one K/V slot per step
// (K_j with V_{j-1}), items claimed dynamically, longest first.
//   warps 0-3 / 4-7  softmax, snapshot and epilogue of tile A / B
//   warp 8           item claimer and TMA producer
//   warp 9           TMEM allocator and MMA issuer
//   warps 10-11      idle (third warpgroup of the register split)
// TMEM: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).  The O_SWA
// snapshot (fp32, normalised) goes to a workspace row that the epilogue reads
// back a few microseconds later (L2-resident): ||o_FULL - o_SWA||^2 and the
// gated output come from the fp32 values.

#include "ptx.cuh"
#include "swiattn_internal.h"

#include <cuda_bf16.h>
#include <math.h>

namespace swi {
namespace {

constexpr int kStages = 2;
constexpr int kThreads = 384;
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsOther = 72;
constexpr int kTileBytes = kBM * kHD * 2;    // 32 KiB
constexpr int kHalfBytes = kTileBytes / 2;   // 16 KiB
constexpr int kSched = 4;
constexpr int kStageBytesPerWarp = 32 * 64 * 2;   // 32 rows x 64 bf16 columns

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffStage = kOffV + kStages * kTileBytes;
constexpr int kOffBar = kOffStage + 8 * kStageBytesPerWarp;

enum {
    BAR_Q_FULL = 0,                        // [2] per tile
    BAR_Q_EMPTY = BAR_Q_FULL + 2,          // [2]
    BAR_KV_FULL = BAR_Q_EMPTY + 2,         // [kStages]: slot of step g holds K_j and V_{j-1}
    BAR_KV_EMPTY = BAR_KV_FULL + kStages,  // [kStages]
    BAR_S_FULL = BAR_KV_EMPTY + kStages,   // [2]
    BAR_P_FULL = BAR_S_FULL + 2,           // [2]
    BAR_O_FULL = BAR_P_FULL + 2,           // [2]
    BAR_O_FREE = BAR_O_FULL + 2,           // [2]
    BAR_SNAP = BAR_O_FREE + 2,             // [2] a tile's window PVs are complete
    BAR_SCHED_FULL = BAR_SNAP + 2,         // [kSched]
    BAR_SCHED_EMPTY = BAR_SCHED_FULL + kSched,
    BAR_DRAIN = BAR_SCHED_EMPTY + kSched,
    BAR_COUNT
};
constexpr uint32_t kSchedConsumers = 1 + 8;

constexpr int kOffSched = kOffBar + BAR_COUNT * 8;
constexpr int kOffMisc = kOffSched + kSched * 4;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int x) { return x ? 128u : 0u; }
__device__ __forceinline__ uint32_t col_o(int x) { return x ? 384u : 256u; }

constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, kHD, false, true);

struct DuParams {
    CUtensorMap tm_q, tm_k, tm_v;
    int* next_item;          // work counter, zeroed before the launch
    const float* logits;
    __nv_bfloat16* o_full;
    __nv_bfloat16* o_swa;
    __nv_bfloat16* o_gated;  // nullable
    float* lse_gated;        // [B,N,Hq] lse of the gated output, nullable
    float* snap;             // [B,N,Hq,128] fp32 O_SWA rows (scratch)
    float* mse_part;         // [B,N,Hq]
    unsigned int* err;
    int B, N, Hq, Hkv, W, NP, n_items;
    float scale_log2;
};

struct Plan {
    int b, h, kvh, q0;
    int nrows[2];
    int kvw, n1, n2;      // window sweep: first key, blocks; far sweep: blocks (from key 0)
    int jw0[2], jw1[2];   // window run of each tile (jw0 > jw1: tile empty)
    int jf1[2];           // far run of each tile: blocks n1 .. n1 + jf1 (-1: none)
};

__device__ __forceinline__ Plan make_plan(const DuParams& p, int idx) {
    Plan pl;
    const int per = p.B * p.Hq;
    const int pair = p.NP - 1 - idx / per;   // latest rows (longest) first
    const int rem = idx % per;
    pl.b = rem / p.Hq;
    pl.h = rem % p.Hq;
    pl.kvh = pl.h / (p.Hq / p.Hkv);
    pl.q0 = pair * 2 * kBM;
    pl.kvw = max(0, pl.q0 - p.W + 1);
    int n1 = 0, n2 = 0;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int r0 = pl.q0 + x * kBM;
        const int nr = max(0, min(kBM, p.N - r0));
        pl.nrows[x] = nr;
        if (nr > 0) {
            const int lo = max(0, r0 - p.W + 1), hi = r0 + nr - 1;
            pl.jw0[x] = (lo - pl.kvw) / kBN;
            pl.jw1[x] = (hi - pl.kvw) / kBN;
            n1 = max(n1, pl.jw1[x] + 1);
            const int fh = hi - p.W;
            pl.jf1[x] = fh >= 0 ? fh / kBN : -1;
            n2 = max(n2, pl.jf1[x] + 1);
        } else {
            pl.jw0[x] = 1;
            pl.jw1[x] = 0;
            pl.jf1[x] = -1;
        }
    }
    pl.n1 = n1;
    pl.n2 = n2;
    return pl;
}

__device__ __forceinline__ bool tile_active(const Plan& pl, int x) { return pl.nrows[x] > 0; }
__device__ __forceinline__ bool blk_active(const Plan& pl, int x, int j) {
    return (j >= pl.jw0[x] && j <= pl.jw1[x]) || (j >= pl.n1 && j - pl.n1 <= pl.jf1[x]);
}
__device__ __forceinline__ int first_blk(const Plan& pl, int x) { return pl.jw0[x]; }
__device__ __forceinline__ int last_blk(const Plan& pl, int x) {
    return pl.jf1[x] >= 0 ? pl.n1 + pl.jf1[x] : pl.jw1[x];
}
__device__ __forceinline__ int blk_key0(const Plan& pl, int j) {
    return j < pl.n1 ? pl.kvw + j * kBN : (j - pl.n1) * kBN;
}

// ----------------------------------------------------------------- roles --

__device__ bool publish_item(const DuParams& p, uint64_t* bar, volatile int* sched, int k,
                             volatile int* abort_flag, int& idx) {
    const int slot = k % kSched;
    const uint32_t par = (static_cast<uint32_t>(k) / kSched) & 1u;
    if (!mbar_wait_w(&bar[BAR_SCHED_EMPTY + slot], par ^ 1u, abort_flag, p.err)) return false;
    int v = 0;
    if ((threadIdx.x & 31) == 0) v = atomicAdd(p.next_item, 1);
    v = __shfl_sync(0xffffffffu, v, 0);
    idx = v < p.n_items ? v : -1;
    if ((threadIdx.x & 31) == 0) {
        sched[slot] = idx;
        mbar_arrive(&bar[BAR_SCHED_FULL + slot]);
    }
    __syncwarp();
    return true;
}

__device__ bool consume_item(const DuParams& p, uint64_t* bar, volatile int* sched, int k,
                             volatile int* abort_flag, int& idx) {
    const int slot = k % kSched;
    const uint32_t par = (static_cast<uint32_t>(k) / kSched) & 1u;
    if (!mbar_wait_w(&bar[BAR_SCHED_FULL + slot], par, abort_flag, p.err)) return false;
    idx = sched[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&bar[BAR_SCHED_EMPTY + slot]);
    return true;
}

__device__ bool producer(const DuParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                         volatile int* abort_flag, uint32_t& g, uint32_t* q_issued) {
    for (int k = 0;; ++k) {
        int idx;
        if (!publish_item(p, bar, sched, k, abort_flag, idx)) return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        const int nblk = pl.n1 + pl.n2;
        auto load_q = [&](int x) -> bool {
            if (!mbar_wait_w(&bar[BAR_Q_EMPTY + x], (q_issued[x] & 1u) ^ 1u, abort_flag, p.err)) return false;
            mbar_arrive_expect_tx_w(&bar[BAR_Q_FULL + x], kTileBytes);
            uint8_t* dst = smem + kOffQ + x * kTileBytes;
            const int row = pl.q0 + x * kBM;
            tma_load_4d_w(dst, &p.tm_q, &bar[BAR_Q_FULL + x], 0, pl.h, row, pl.b);
            tma_load_4d_w(dst + kHalfBytes, &p.tm_q, &bar[BAR_Q_FULL + x], 64, pl.h, row, pl.b);
            ++q_issued[x];
            return true;
        };
        if (tile_active(pl, 0) && !load_q(0)) return false;
        for (int j = 0; j <= nblk; ++j) {
            if (j < nblk && tile_active(pl, 1) && j == first_blk(pl, 1) && !load_q(1)) return false;
            const uint32_t st = g % kStages, ph = (g / kStages) & 1u;
            if (!mbar_wait_w(&bar[BAR_KV_EMPTY + st], ph ^ 1u, abort_flag, p.err)) return false;
            const uint32_t bytes = (j < nblk ? kTileBytes : 0) + (j >= 1 ? kTileBytes : 0);
            mbar_arrive_expect_tx_w(&bar[BAR_KV_FULL + st], bytes);
            if (j < nblk) {
                uint8_t* dst = smem + kOffK + st * kTileBytes;
                const int key0 = blk_key0(pl, j);
                tma_load_4d_w(dst, &p.tm_k, &bar[BAR_KV_FULL + st], 0, pl.kvh, key0, pl.b);
                tma_load_4d_w(dst + kHalfBytes, &p.tm_k, &bar[BAR_KV_FULL + st], 64, pl.kvh, key0, pl.b);
            }
            if (j >= 1) {
                uint8_t* dst = smem + kOffV + st * kTileBytes;
                const int key0 = blk_key0(pl, j - 1);
                tma_load_4d_w(dst, &p.tm_v, &bar[BAR_KV_FULL + st], 0, pl.kvh, key0, pl.b);
                tma_load_4d_w(dst + kHalfBytes, &p.tm_v, &bar[BAR_KV_FULL + st], 64, pl.kvh, key0, pl.b);
            }
            ++g;
        }
    }
    return true;
}

__device__ void drain_loads(uint64_t* full_bars, uint32_t issued) {
    for (uint32_t back = 1; back <= kStages && back <= issued; ++back) {
        const uint32_t it = issued - back;
        mbar_drain(&full_bars[it % kStages], (it / kStages) & 1u);
    }
}

__device__ bool mma_issuer(const DuParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                           uint32_t tmem, volatile int* abort_flag) {
    uint32_t g = 0;
    uint32_t q_cnt[2] = {0, 0}, p_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};

    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, bar, sched, k, abort_flag, idx)) return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        const int nblk = pl.n1 + pl.n2;
        int pend[2] = {-1, -1};
        bool first_pv[2] = {true, true};

        auto issue_pv = [&](int x, int jj, uint32_t sV) -> bool {
            if (!mbar_wait_w(&bar[BAR_P_FULL + x], p_cnt[x] & 1u, abort_flag, p.err)) return false;
            ++p_cnt[x];
            if (first_pv[x]) {
                if (!mbar_wait_w(&bar[BAR_O_FREE + x], (o_cnt[x] & 1u) ^ 1u, abort_flag, p.err))
                    return false;
                ++o_cnt[x];
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
                const uint64_t bdesc = sdesc_sw128(sV + kk * 16 * 128, kHalfBytes, 1024);
                umma_bf16_ts_w(tmem + col_o(x), tmem + col_s(x) + kk * 8, bdesc, kIdescO,
                               (first_pv[x] && kk == 0) ? 0u : 1u);
            }
            first_pv[x] = false;
            if (jj == pl.jw1[x] && pl.jf1[x] >= 0) umma_commit_w(&bar[BAR_SNAP + x]);
            if (jj == last_blk(pl, x)) umma_commit_w(&bar[BAR_O_FULL + x]);
            return true;
        };

        for (int j = 0; j <= nblk; ++j) {
            const uint32_t st = g % kStages, ph = (g / kStages) & 1u;
            if (!mbar_wait_w(&bar[BAR_KV_FULL + st], ph, abort_flag, p.err)) return false;
            tc_fence_after();
            const uint32_t sK = smem_u32(smem + kOffK + st * kTileBytes);
            const uint32_t sV = smem_u32(smem + kOffV + st * kTileBytes);
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                // PV of the previous block first: P_x lives in S_x's columns.
                if (pend[x] >= 0) {
                    if (!issue_pv(x, pend[x], sV)) return false;
                    pend[x] = -1;
                }
                if (j < nblk && tile_active(pl, x) && blk_active(pl, x, j)) {
                    if (j == first_blk(pl, x)) {
                        if (!mbar_wait_w(&bar[BAR_Q_FULL + x], q_cnt[x] & 1u, abort_flag, p.err))
                            return false;
                        ++q_cnt[x];
                        tc_fence_after();
                    }
                    const uint32_t sQ = smem_u32(smem + kOffQ + x * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kHD / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                        umma_bf16_w(tmem + col_s(x), sdesc_sw128(sQ + off, 16, 1024),
                                    sdesc_sw128(sK + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
                    }
                    umma_commit_w(&bar[BAR_S_FULL + x]);
                    if (j == last_blk(pl, x)) umma_commit_w(&bar[BAR_Q_EMPTY + x]);
                    pend[x] = j;
                }
            }
            umma_commit_w(&bar[BAR_KV_EMPTY + st]);
            ++g;
        }
    }
    return true;
}

// One warp's 32 rows x 64 bf16 columns (column half hh) to global memory in
// whole 128-byte row segments: each lane stages its row (pk: 32 packed pairs)
// in the warp's shared-memory area, then every store instruction writes four
// rows.  out_row / wflag are per lane (its row's destination and whether to
// write it).  Warp-collective.
__device__ __forceinline__ void store_half_staged(uint32_t stg, int lane, const uint32_t* pk,
                                                  unsigned long long out_row, int wflag,
                                                  __nv_bfloat16* base, int hh) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
        st_shared_v4(stg + lane * 128 + ((((uint32_t)u) ^ ((uint32_t)lane & 7u)) << 4), pk[4 * u],
                     pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int row = it * 4 + (lane >> 3);
        const uint32_t u = lane & 7;
        const unsigned long long orow = __shfl_sync(0xffffffffu, out_row, row);
        const int wf = __shfl_sync(0xffffffffu, wflag, row);
        const uint4 val = ld_shared_v4(stg + row * 128 + ((u ^ ((uint32_t)row & 7u)) << 4));
        if (wf) *reinterpret_cast<uint4*>(base + orow * kHD + hh * 64 + u * 8) = val;
    }
    __syncwarp();
}

// One key block of tile x for its softmax warp: S from TMEM, masked maximum
// over the visible columns [a, e], running max / rescale, P (bf16) back over
// S, row sum.  Returns false when a wait timed out.
__device__ __forceinline__ bool softmax_block(const DuParams& p, uint64_t* bar, volatile int* abort_flag,
                                              int x, uint32_t tS, uint32_t tO, int a, int e,
                                              uint32_t& s_cnt, float& m2, float& l) {
    const float sl = p.scale_log2;
    if (!mbar_wait_w(&bar[BAR_S_FULL + x], s_cnt & 1u, abort_flag, p.err)) return false;
    ++s_cnt;
    tc_fence_after();
    uint32_t sr[128];
    tmem_ld32(tS + 0, sr);
    tmem_ld32(tS + 32, sr + 32);
    tmem_ld32(tS + 64, sr + 64);
    tmem_ld32(tS + 96, sr + 96);
    tmem_ld_wait();
    float* s = reinterpret_cast<float*>(sr);
    // Warp-uniform classification (every lane votes, the branches follow the
    // votes, so a warp never runs two paths): a one-sided mask (visible
    // c <= e or c >= a for the whole warp) costs one compare and one select
    // per column; the maximum is the three-input tree of a full block.
    const bool all_full = __all_sync(0xffffffffu, a <= 0 && e >= kBN - 1);
    const bool all_pre = __all_sync(0xffffffffu, a <= 0);
    const bool all_suf = __all_sync(0xffffffffu, e >= kBN - 1);
    float m8[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) m8[t] = -INFINITY;
    if (!all_full) {
        if (all_pre) {
#pragma unroll
            for (int cc = 0; cc < kBN; ++cc) s[cc] = cc <= e ? s[cc] : -INFINITY;
        } else if (all_suf) {
#pragma unroll
            for (int cc = 0; cc < kBN; ++cc) s[cc] = cc >= a ? s[cc] : -INFINITY;
        } else {
            const uint32_t span = static_cast<uint32_t>(e - a);
#pragma unroll
            for (int cc = 0; cc < kBN; ++cc) {
                const bool ok = static_cast<uint32_t>(cc - a) <= span && e >= a;
                s[cc] = ok ? s[cc] : -INFINITY;
            }
        }
    }
#pragma unroll
    for (int cc = 0; cc < kBN; cc += 16)
#pragma unroll
        for (int t = 0; t < 8; ++t) m8[t] = fmax3(m8[t], s[cc + 2 * t], s[cc + 2 * t + 1]);
    const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
    // Running max in scaled log2 units; O and l are rescaled only when the max
    // grows by more than 2^8 (p stays <= 256 otherwise).
    const float mnew = fmaxf(m2, mx * sl);
    const bool resc = mnew > m2 + 8.0f;
    float alpha = 1.f;
    if (resc) {
        alpha = ex2_approx(m2 - mnew);
        m2 = mnew;
    }
    // O_x is stable here: S_x(j) completing implies the earlier PV_x did.
    const bool need = resc && l > 0.f;
    if (__any_sync(0xffffffffu, need)) {
        const float f = need ? alpha : 1.f;
        // Sixteen columns at a time: this runs while the block's 128 scores
        // are live, so the narrower load keeps the peak register count down.
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
            uint32_t orr[16];
            tmem_ld16(tO + q8 * 16, orr);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 16; ++t) orr[t] = __float_as_uint(__uint_as_float(orr[t]) * f);
            tmem_st16(tO + q8 * 16, orr);
        }
    }
    const float mb = (m2 == -INFINITY) ? 0.f : m2;
    const float2 sl2 = make_float2(sl, sl), nmb = make_float2(-mb, -mb);
    float2 r4[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) r4[t] = make_float2(0.f, 0.f);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
#pragma unroll
        for (int pp = 0; pp < 32; ++pp) {
            const int cc = hh * 64 + 2 * pp;
            const float2 xv = ffma2(make_float2(s[cc], s[cc + 1]), sl2, nmb);
            float2 pv;
            pv.x = ex2_approx(xv.x);
            pv.y = ex2_approx(xv.y);
            r4[pp & 3] = fadd2(r4[pp & 3], pv);
            pk[pp] = pack_bf16x2(pv.x, pv.y);
        }
        tmem_st32(tS + hh * 32, pk);   // P over the S columns already consumed
    }
    const float2 rs2 = fadd2(fadd2(r4[0], r4[1]), fadd2(r4[2], r4[3]));
    tmem_st_wait();
    l = l * alpha + (rs2.x + rs2.y);
    tc_fence_before();
    mbar_arrive(&bar[BAR_P_FULL + x]);
    return true;
}

__device__ bool softmax_role(const DuParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                             uint32_t tmem, volatile int* abort_flag, int x, int wq, int lane) {
    const int r = wq * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = lane_base + col_s(x);
    const uint32_t tO = lane_base + col_o(x);
    const uint32_t stg = smem_u32(smem + kOffStage + (x * 4 + wq) * kStageBytesPerWarp);
    uint32_t s_cnt = 0, o_cnt = 0, snap_cnt = 0;

    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, bar, sched, k, abort_flag, idx)) return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        if (!tile_active(pl, x)) continue;
        const int i = r < pl.nrows[x] ? pl.q0 + x * kBM + r : -1;
        const unsigned long long out_row =
            (i >= 0) ? (((unsigned long long)pl.b * p.N + i) * p.Hq + pl.h) : 0ull;
        const int wflag = i >= 0 ? 1 : 0;
        const bool has_far = pl.jf1[x] >= 0;
        float m2 = -INFINITY, l = 0.f;
        float lse_swa = 0.f;   // natural-log lse of the window branch (set at the snapshot)

        // Window run: keys [max(0, i-W+1), i].
        for (int j = pl.jw0[x]; j <= pl.jw1[x]; ++j) {
            const int key0 = pl.kvw + j * kBN;
            const int a = (i >= 0) ? max(0, i - p.W + 1) - key0 : 1;
            const int e = (i >= 0) ? i - key0 : 0;
            if (!softmax_block(p, bar, abort_flag, x, tS, tO, a, e, s_cnt, m2, l)) return false;
        }
        if (has_far) {
            // Every window PV of this tile is complete: O/l is O_SWA.  Keep it
            // (fp32) for the epilogue and write it.
            if (!mbar_wait_w(&bar[BAR_SNAP + x], snap_cnt & 1u, abort_flag, p.err)) return false;
            ++snap_cnt;
            tc_fence_after();
            const float inv = (l > 0.f) ? 1.f / l : 0.f;
            lse_swa = (m2 + __log2f(l)) * 0.69314718055994531f;
            float* snap_row = p.snap + out_row * kHD;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t pk[32];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t orr[32];
                    tmem_ld32(tO + hh * 64 + q * 32, orr);
                    tmem_ld_wait();
                    float* v = reinterpret_cast<float*>(orr);
#pragma unroll
                    for (int t = 0; t < 32; ++t) v[t] *= inv;
#pragma unroll
                    for (int t = 0; t < 16; ++t) pk[q * 16 + t] = pack_bf16x2(v[2 * t], v[2 * t + 1]);
                    if (i >= 0) {
                        float4* dst = reinterpret_cast<float4*>(snap_row + hh * 64 + q * 32);
#pragma unroll
                        for (int t = 0; t < 8; ++t)
                            dst[t] = make_float4(v[4 * t], v[4 * t + 1], v[4 * t + 2], v[4 * t + 3]);
                    }
                }
                store_half_staged(stg, lane, pk, out_row, wflag, p.o_swa, hh);
            }
        }
        // Far run: keys [0, i-W].
        for (int j = 0; j <= pl.jf1[x]; ++j) {
            const int key0 = j * kBN;
            const int a = (i >= 0) ? -key0 : 1;
            const int e = (i >= 0) ? i - p.W - key0 : 0;
            if (!softmax_block(p, bar, abort_flag, x, tS, tO, a, e, s_cnt, m2, l)) return false;
        }

        // Epilogue: O_FULL = O/l; O_SWA from the snapshot (or O_FULL when the
        // tile has no key beyond the window); squared distance; gated output.
        if (!mbar_wait_w(&bar[BAR_O_FULL + x], o_cnt & 1u, abort_flag, p.err)) return false;
        ++o_cnt;
        tc_fence_after();
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const bool gated_full = (i >= 0) ? (p.logits[(size_t)pl.b * p.N + i] > 0.f) : false;
        const float* snap_row = p.snap + out_row * kHD;
        float mse = 0.f;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t pf[32], pg[32];   // O_FULL and gated output, bf16 pairs
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t orr[32];
                tmem_ld32(tO + hh * 64 + q * 32, orr);
                tmem_ld_wait();
                float* fv = reinterpret_cast<float*>(orr);
#pragma unroll
                for (int t = 0; t < 32; ++t) fv[t] *= inv;
                float sv[32];
                if (has_far && i >= 0) {
                    const float4* src = reinterpret_cast<const float4*>(snap_row + hh * 64 + q * 32);
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const float4 v4 = src[t];
                        sv[4 * t] = v4.x;
                        sv[4 * t + 1] = v4.y;
                        sv[4 * t + 2] = v4.z;
                        sv[4 * t + 3] = v4.w;
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) sv[t] = fv[t];
                }
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const float dlt = fv[t] - sv[t];
                    mse = fmaf(dlt, dlt, mse);
                }
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    pf[q * 16 + t] = pack_bf16x2(fv[2 * t], fv[2 * t + 1]);
                    pg[q * 16 + t] = gated_full ? pf[q * 16 + t] : pack_bf16x2(sv[2 * t], sv[2 * t + 1]);
                }
            }
            store_half_staged(stg, lane, pf, out_row, wflag, p.o_full, hh);
            if (!has_far) store_half_staged(stg, lane, pf, out_row, wflag, p.o_swa, hh);
            if (p.o_gated) store_half_staged(stg, lane, pg, out_row, wflag, p.o_gated, hh);
        }
        if (i >= 0) p.mse_part[out_row] = mse;
        if (i >= 0 && p.lse_gated) {
            const float lse_full = (m2 + __log2f(l)) * 0.69314718055994531f;
            p.lse_gated[out_row] = (gated_full || !has_far) ? lse_full : lse_swa;
        }
        tc_fence_before();
        mbar_arrive(&bar[BAR_O_FREE + x]);
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) dual_kernel(const __grid_constant__ DuParams p) {
    // The epilogue kernel after it is a programmatic dependent launch: it may
    // be scheduled now and waits for this grid before reading the partials.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
    volatile int* sched = reinterpret_cast<volatile int*>(smem + kOffSched);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bar[BAR_Q_FULL + x], 1);
            mbar_init(&bar[BAR_Q_EMPTY + x], 1);
            mbar_init(&bar[BAR_S_FULL + x], 1);
            mbar_init(&bar[BAR_P_FULL + x], kBM);
            mbar_init(&bar[BAR_O_FULL + x], 1);
            mbar_init(&bar[BAR_O_FREE + x], kBM);
            mbar_init(&bar[BAR_SNAP + x], 1);
        }
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&bar[BAR_KV_FULL + st], 1);
            mbar_init(&bar[BAR_KV_EMPTY + st], 1);
        }
        for (int st = 0; st < kSched; ++st) {
            mbar_init(&bar[BAR_SCHED_FULL + st], 1);
            mbar_init(&bar[BAR_SCHED_EMPTY + st], kSchedConsumers);
        }
        mbar_init(&bar[BAR_DRAIN], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 8) {
        warpgroup_reg_inc<kRegsSoftmax>();
        softmax_role(p, smem, bar, sched, tmem, abort_flag, warp >> 2, warp & 3, lane);
    } else {
        warpgroup_reg_dec<kRegsOther>();
    }
    if (warp == 8) {
        if (lane == 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
        }
        __syncwarp();
        uint32_t g = 0, q_issued[2] = {0, 0};
        if (!producer(p, smem, bar, sched, abort_flag, g, q_issued)) {
            drain_loads(&bar[BAR_KV_FULL], g);
            for (int x = 0; x < 2; ++x)
                if (q_issued[x]) mbar_drain(&bar[BAR_Q_FULL + x], (q_issued[x] - 1) & 1u);
        }
        __syncwarp();
    } else if (warp == 9) {
        mma_issuer(p, smem, bar, sched, tmem, abort_flag);
        umma_commit_w(&bar[BAR_DRAIN]);
        mbar_drain(&bar[BAR_DRAIN], 0);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_dual_tc(const TcAttnArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
    DuParams p;
    memset(&p, 0, sizeof(p));
    const uint64_t N = a.N, B = a.B;
    bool ok = make_tmap_4d_bf16(&p.tm_q, a.q, kHD, a.Hq, N, B, 64, kBM) &&
              make_tmap_4d_bf16(&p.tm_k, a.k, kHD, a.Hkv, N, B, 64, kBN) &&
              make_tmap_4d_bf16(&p.tm_v, a.v, kHD, a.Hkv, N, B, 64, kBN);
    if (!ok) return cudaErrorInvalidValue;
    p.next_item = a.counter;
    p.logits = a.logits;
    p.o_full = static_cast<__nv_bfloat16*>(a.o);
    p.o_swa = static_cast<__nv_bfloat16*>(a.o_swa);
    p.o_gated = static_cast<__nv_bfloat16*>(a.o_gated);
    p.lse_gated = a.lse;
    p.snap = a.snap;
    p.mse_part = a.mse_part;
    p.err = err;
    p.B = a.B;
    p.N = a.N;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.W = a.W;
    p.NP = (a.N + 2 * kBM - 1) / (2 * kBM);
    p.n_items = p.NP * a.B * a.Hq;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    static std::atomic<uint64_t> smem_allowed{0};
    cudaError_t e = allow_dynamic_smem(dual_kernel, kSmemBytes, smem_allowed);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(a.counter, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
    prof_start(s);
    dual_kernel<<<num_sms, kThreads, kSmemBytes, s>>>(p);
    prof_stop(s);
    return cudaGetLastError();
}

cudaError_t dual_set_wait_limit(uint64_t ns) { return set_wait_limit_of_unit(ns); }

}  // namespace swi
