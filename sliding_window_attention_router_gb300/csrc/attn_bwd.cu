// Backward of routed attention on the 5th-generation tensor cores (sm_103a).
//
// Chain rule through each row's softmax over its visited keys (the row's
// gradient reaches only the branch its hard straight-through gate selected;
// SwiAttn report, section 2):
//   p_ij = exp(scale q_i.k_j - lse_i),  dS_ij = p_ij (dO_i.v_j - D_i),
//   D_i = dO_i.O_i,  dV_j = sum_i p_ij dO_i,  dK_j = scale sum_i dS_ij q_i,
//   dQ_i = scale sum_j dS_ij k_j.
// Two persistent kernels, no atomics (results are bitwise repeatable):
//
// dK/dV (key-stationary).  An item is one 128-key block of one (b, kv head);
// it visits, for every query head of the GQA group, the band query tiles whose
// window reaches the block (every row's window part, [i-W+1, i]) and the far
// tiles of compacted routed rows whose prefix [0, i-W] reaches it.  Per tile:
//   S^T  = K Q^T      (SS)   -> softmax warps: P^T = exp2(S^T*scale*log2e - lse2)
//   dP^T = V dO^T     (SS)   -> softmax warps: dS^T = P^T (dP^T - D)
//   dV  += P^T dO     (TS: P^T read from TMEM as bf16)
//   dK  += dS^T Q     (TS: dS^T read from TMEM as bf16)
// TMEM: S^T [0,128) (P^T over it), dP^T [128,256) (dS^T over it), dV [256,384),
// dK [384,512).  The MMA warp issues dV(t), S^T(t+1), dK(t), dP^T(t+1), so the
// tensor core works on the next tile while the softmax warps finish this one.
//
// dQ (query-stationary).  An item is one 128-row query tile of one (b, query
// head): a band tile walks its window keys, a far tile of compacted routed
// rows walks [0, max i] (so every dQ row has exactly one writer; band tiles
// skip their far rows).  Per key block:
//   S = Q K^T, dP = dO V^T (SS) -> dS = P (dP - D) -> dQ += dS K (TS).
// TMEM: S ring [0,256) (dS over it), dP [256,384), dQ [384,512).
//
// Roles (384 threads, as in the forward): warps 0-7 softmax and epilogue;
// warp w serves TMEM lanes 32*(w%4).. (key rows, or query rows) and column
// half w/4 of each 128-column tile; warp 8 claims items and issues TMA loads;
// warp 9 allocates TMEM and issues the MMAs; warps 10-11 complete the third
// warpgroup for the register split (216 / 72).

#include "ptx.cuh"
#include "swiattn_internal.h"

#include <cuda_bf16.h>
#include <climits>
#include <math.h>

namespace swi {
namespace {

constexpr int kThreads = 384;
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsOther = 72;
constexpr int kTileBytes = kBM * kHD * 2;   // 32 KiB
constexpr int kHalfBytes = kTileBytes / 2;
constexpr int kRowBytes = kBM * 4;          // 128 fp32 / int32 per tile
constexpr int kSched = 4;
constexpr uint32_t kSchedConsumers = 1 + 8;  // MMA warp + softmax warps
constexpr uint32_t kSoftmaxThreads = 256;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescSS = idesc_bf16_f32(kBM, kBN, false, false);   // both K-major
constexpr uint32_t kIdescTS = idesc_bf16_f32(kBM, kHD, false, true);    // B MN-major

struct BwdParams {
    CUtensorMap tm_q, tm_qc, tm_do, tm_doc, tm_k, tm_v;
    const BwdItem* items;
    const int* n_items;
    int* next_item;
    const int* routed_count;
    const int* rowidx;
    const float* d_band;
    const float* l_band;
    const float* d_far;
    const float* l_far;
    const uint8_t* gate;
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    unsigned int* err;
    int B, N, Npad, Hq, Hkv, W;
    float scale, scale_log2;
};

// 1-D bulk copy global -> shared completing on an mbarrier (both addresses
// 16-byte aligned, size a multiple of 16), issued by one elected lane.
__device__ __forceinline__ void bulk_load_w(void* smem_dst, const void* src, uint32_t bytes,
                                            uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
        ::"r"(smem_u32(smem_dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ BwdItem load_item(const BwdParams& p, int idx) {
    const int4* src = reinterpret_cast<const int4*>(p.items + idx);
    const int4 a = src[0], b = src[1];
    BwdItem it;
    it.kind = a.x;
    it.b = a.y;
    it.h = a.z;
    it.t = a.w;
    it.a0 = b.x;
    it.a1 = b.y;
    it.a2 = b.z;
    it.cost = b.w;
    return it;
}

// ---------------------------------------------------------- item ring ------
__device__ bool publish_item(const BwdParams& p, uint64_t* full, uint64_t* empty,
                             volatile int* sched, int k, int n, volatile int* abort_flag,
                             int& idx) {
    const int slot = k % kSched;
    const uint32_t par = (static_cast<uint32_t>(k) / kSched) & 1u;
    if (!mbar_wait_w(&empty[slot], par ^ 1u, abort_flag, p.err)) return false;
    int v = 0;
    if ((threadIdx.x & 31) == 0) v = atomicAdd(p.next_item, 1);
    v = __shfl_sync(0xffffffffu, v, 0);
    idx = v < n ? v : -1;
    if ((threadIdx.x & 31) == 0) {
        sched[slot] = idx;
        mbar_arrive(&full[slot]);
    }
    __syncwarp();
    return true;
}

__device__ bool consume_item(const BwdParams& p, uint64_t* full, uint64_t* empty,
                             volatile int* sched, int k, volatile int* abort_flag, int& idx) {
    const int slot = k % kSched;
    const uint32_t par = (static_cast<uint32_t>(k) / kSched) & 1u;
    if (!mbar_wait_w(&full[slot], par, abort_flag, p.err)) return false;
    idx = sched[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[slot]);
    return true;
}

__device__ __forceinline__ void load_tile_pair(const CUtensorMap* map, uint8_t* dst, uint64_t* bar,
                                               int h, int row, int b) {
    tma_load_4d_w(dst, map, bar, 0, h, row, b);
    tma_load_4d_w(dst + kHalfBytes, map, bar, 64, h, row, b);
}

// K-step kk of a 128-deep K-major operand in a two-half SW128 tile.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
    // The start address is the descriptor's low field (16-byte units, no carry
    // within shared memory): the tile's descriptor plus the step's offset, so
    // the per-step descriptors of one tile share one computed base.
    return sdesc_sw128(tile, 16, 1024) +
           static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
}
// K-step kk (16 rows) of an MN-major B operand (rows = K, 128 columns = N).
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
    return sdesc_sw128(tile, kHalfBytes, 1024) + static_cast<uint64_t>((kk * 16 * 128) >> 4);
}
// TMEM column of K-step kk of a bf16 operand packed per column half: keys or
// queries 0-63 at columns [0, 32), 64-127 at [64, 96) of the 128-column block.
__device__ __forceinline__ uint32_t packed_col(int kk) {
    return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8);
}

// After an abort: waits (bounded) for the loads still in flight on a ring of
// `slots` full-barriers, of which `issued` have been armed so far.
__device__ __forceinline__ void drain_ring(uint64_t* bars, uint32_t slots, uint32_t issued) {
    for (uint32_t back = 1; back <= slots && back <= issued; ++back) {
        const uint32_t it = issued - back;
        mbar_drain(&bars[it % slots], (it / slots) & 1u);
    }
}

// Converts 64 fp32 values to bf16 pairs and stores them (128 bytes) at dst.
__device__ __forceinline__ void store_row64(__nv_bfloat16* dst, const uint32_t* v, float mul) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]) * mul, __uint_as_float(v[8 * u + 1]) * mul);
        w.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul);
        w.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul);
        w.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul);
        d4[u] = w;
    }
}

// Masks columns outside [a, e] of this warp's 64-column half (column c of
// the tile is x[c - c0]) by setting the exponent argument to -inf.  Must be
// reached by the whole warp: it votes for a one-sided mask (visible c <= e,
// or c >= a, for every lane), which costs one compare and one select per
// column; the branches follow the votes.
__device__ __forceinline__ void mask_half(float* x, int a, int e, int c0) {
    const bool all_pre = __all_sync(0xffffffffu, a <= c0);
    const bool all_suf = __all_sync(0xffffffffu, e >= c0 + 63);
    if (all_pre) {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = c0 + c <= e ? x[c] : -INFINITY;
    } else if (all_suf) {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = c0 + c >= a ? x[c] : -INFINITY;
    } else {
        const uint32_t span = static_cast<uint32_t>(e - a);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const bool ok = static_cast<uint32_t>(c0 + c - a) <= span && e >= a;
            x[c] = ok ? x[c] : -INFINITY;
        }
    }
}

// =================================================================== dK/dV ==
namespace kv {

// Query tiles live from S^T(t) to dK += dS^T(t) Q(t): three slots keep their
// loads a tile and more ahead; dO tiles (with the tile's per-column lse and D)
// two slots.  The tiles fill 224 KiB; the kernel requires the dynamic shared
// memory base to be 1024-byte aligned (it is: the window's first KiB is
// reserved) and checks it instead of padding.
constexpr int kQSlots = 3;
constexpr int kDSlots = 2;
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kOffQ = kOffV + kTileBytes;                 // [kQSlots] query tiles
constexpr int kOffDO = kOffQ + kQSlots * kTileBytes;      // [kDSlots] dO tiles
constexpr int kOffL = kOffDO + kDSlots * kTileBytes;      // [kDSlots][128] lse * log2 e per column
constexpr int kOffD = kOffL + kDSlots * kRowBytes;        // [kDSlots][128] D per column
constexpr int kOffBar = kOffD + kDSlots * kRowBytes;

enum {
    BAR_K_FULL = 0,
    BAR_K_EMPTY,
    BAR_V_FULL,
    BAR_V_EMPTY,
    BAR_Q_FULL,                             // [kQSlots]
    BAR_Q_EMPTY = BAR_Q_FULL + kQSlots,     // [kQSlots]
    BAR_DO_FULL = BAR_Q_EMPTY + kQSlots,    // [kDSlots]
    BAR_DO_EMPTY = BAR_DO_FULL + kDSlots,   // [kDSlots]
    BAR_S_FULL = BAR_DO_EMPTY + kDSlots,
    BAR_DP_FULL,
    BAR_P_FULL,
    BAR_DS_FULL,
    BAR_ACC_FULL,
    BAR_ACC_FREE,
    BAR_SCHED_FULL,                          // [kSched]
    BAR_SCHED_EMPTY = BAR_SCHED_FULL + kSched,
    BAR_DRAIN = BAR_SCHED_EMPTY + kSched,
    BAR_COUNT
};
constexpr int kOffSched = kOffBar + BAR_COUNT * 8;
constexpr int kOffMisc = kOffSched + kSched * 4;
constexpr int kSmemBytes = kOffMisc + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Plan {
    int b, kvh, k0, G, nband, ft0, nfar, ntiles;
};

__device__ __forceinline__ Plan make_plan(const BwdParams& p, int idx) {
    const BwdItem it = load_item(p, idx);
    Plan pl;
    pl.b = it.b;
    pl.kvh = it.h;
    pl.k0 = it.t * kBN;
    pl.G = p.Hq / p.Hkv;
    pl.nband = it.a0;
    pl.ft0 = it.a1;
    pl.nfar = it.a2 - it.a1;
    pl.ntiles = pl.G * (pl.nband + pl.nfar);
    return pl;
}

struct Tile {
    int h, row0;
    bool far;
};

__device__ __forceinline__ Tile tile_of(const Plan& pl, int u) {
    const int per = pl.nband + pl.nfar;
    const int g = u / per, r = u - g * per;
    Tile t;
    t.h = pl.kvh * pl.G + g;
    t.far = r >= pl.nband;
    t.row0 = t.far ? (pl.ft0 + r - pl.nband) * kBM : pl.k0 + r * kBM;
    return t;
}

// Loads issued so far on each ring of the dK/dV producer (a drain after an
// abort waits for the last one of each ring that can still be in flight).
struct KvIssued {
    uint32_t q, d, k, v;
};

__device__ bool producer(const BwdParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                         volatile int* abort_flag, KvIssued& n_is) {
    const int n = p.n_items[0];
    for (int k = 0;; ++k) {
        int idx;
        if (!publish_item(p, &bar[BAR_SCHED_FULL], &bar[BAR_SCHED_EMPTY], sched, k, n,
                          abort_flag, idx))
            return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        if (!mbar_wait_w(&bar[BAR_K_EMPTY], (n_is.k & 1u) ^ 1u, abort_flag, p.err)) return false;
        mbar_arrive_expect_tx_w(&bar[BAR_K_FULL], kTileBytes);
        load_tile_pair(&p.tm_k, smem + kOffK, &bar[BAR_K_FULL], pl.kvh, pl.k0, pl.b);
        ++n_is.k;
        if (!mbar_wait_w(&bar[BAR_V_EMPTY], (n_is.v & 1u) ^ 1u, abort_flag, p.err)) return false;
        mbar_arrive_expect_tx_w(&bar[BAR_V_FULL], kTileBytes);
        load_tile_pair(&p.tm_v, smem + kOffV, &bar[BAR_V_FULL], pl.kvh, pl.k0, pl.b);
        ++n_is.v;
        for (int u = 0; u < pl.ntiles; ++u) {
            const Tile t = tile_of(pl, u);
            const uint32_t qs = n_is.q % kQSlots, qph = (n_is.q / kQSlots) & 1u;
            if (!mbar_wait_w(&bar[BAR_Q_EMPTY + qs], qph ^ 1u, abort_flag, p.err)) return false;
            mbar_arrive_expect_tx_w(&bar[BAR_Q_FULL + qs], kTileBytes);
            load_tile_pair(t.far ? &p.tm_qc : &p.tm_q, smem + kOffQ + qs * kTileBytes,
                           &bar[BAR_Q_FULL + qs], t.h, t.row0, pl.b);
            ++n_is.q;
            const uint32_t ds = n_is.d % kDSlots, dph = (n_is.d / kDSlots) & 1u;
            if (!mbar_wait_w(&bar[BAR_DO_EMPTY + ds], dph ^ 1u, abort_flag, p.err)) return false;
            uint64_t* fb = &bar[BAR_DO_FULL + ds];
            mbar_arrive_expect_tx_w(fb, kTileBytes + 2 * kRowBytes);
            load_tile_pair(t.far ? &p.tm_doc : &p.tm_do, smem + kOffDO + ds * kTileBytes, fb, t.h,
                           t.row0, pl.b);
            const size_t stat = ((size_t)pl.b * p.Hq + t.h) * p.Npad + t.row0;
            bulk_load_w(smem + kOffL + ds * kRowBytes, (t.far ? p.l_far : p.l_band) + stat,
                        kRowBytes, fb);
            bulk_load_w(smem + kOffD + ds * kRowBytes, (t.far ? p.d_far : p.d_band) + stat,
                        kRowBytes, fb);
            ++n_is.d;
        }
    }
    return true;
}

__device__ bool mma_issuer(const BwdParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                           uint32_t tmem, volatile int* abort_flag) {
    const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;
    const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
    uint32_t g = 0, kv_cnt = 0, acc_cnt = 0;

    // Tile c (a running count over items): query slot c % kQSlots, dO slot
    // c % kDSlots.
    auto issue_s = [&](uint32_t c) -> bool {   // S^T = K Q^T
        const uint32_t qs = c % kQSlots;
        if (!mbar_wait_w(&bar[BAR_Q_FULL + qs], (c / kQSlots) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t sQ = smem_u32(smem + kOffQ + qs * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk)
            umma_bf16_w(tS, kmajor_desc(sK, kk), kmajor_desc(sQ, kk), kIdescSS, kk > 0 ? 1u : 0u);
        umma_commit_w(&bar[BAR_S_FULL]);
        return true;
    };
    auto issue_dp = [&](uint32_t c) -> bool {   // dP^T = V dO^T
        const uint32_t ds = c % kDSlots;
        if (!mbar_wait_w(&bar[BAR_DO_FULL + ds], (c / kDSlots) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t sD = smem_u32(smem + kOffDO + ds * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk)
            umma_bf16_w(tDP, kmajor_desc(sV, kk), kmajor_desc(sD, kk), kIdescSS, kk > 0 ? 1u : 0u);
        umma_commit_w(&bar[BAR_DP_FULL]);
        return true;
    };

    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, &bar[BAR_SCHED_FULL], &bar[BAR_SCHED_EMPTY], sched, k, abort_flag, idx))
            return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        const int T = pl.ntiles;
        if (!mbar_wait_w(&bar[BAR_K_FULL], kv_cnt & 1u, abort_flag, p.err)) return false;
        if (!mbar_wait_w(&bar[BAR_V_FULL], kv_cnt & 1u, abort_flag, p.err)) return false;
        ++kv_cnt;
        if (!issue_s(g)) return false;
        if (T == 1) umma_commit_w(&bar[BAR_K_EMPTY]);
        if (!issue_dp(g)) return false;
        if (T == 1) umma_commit_w(&bar[BAR_V_EMPTY]);
        for (int t = 0; t < T; ++t) {
            const uint32_t cur = g + t;
            if (!mbar_wait_w(&bar[BAR_P_FULL], cur & 1u, abort_flag, p.err)) return false;
            if (t == 0 && !mbar_wait_w(&bar[BAR_ACC_FREE], (acc_cnt & 1u) ^ 1u, abort_flag, p.err))
                return false;
            tc_fence_after();
            const uint32_t sD = smem_u32(smem + kOffDO + (cur % kDSlots) * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kBM / 16; ++kk)   // dV += P^T dO
                umma_bf16_ts_w(tDV, tS + packed_col(kk), mnmajor_desc(sD, kk), kIdescTS,
                               (t > 0 || kk > 0) ? 1u : 0u);
            if (t + 1 < T) {
                if (!issue_s(cur + 1)) return false;
                if (t + 2 == T) umma_commit_w(&bar[BAR_K_EMPTY]);
            }
            if (!mbar_wait_w(&bar[BAR_DS_FULL], cur & 1u, abort_flag, p.err)) return false;
            tc_fence_after();
            const uint32_t sQ = smem_u32(smem + kOffQ + (cur % kQSlots) * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kBM / 16; ++kk)   // dK += dS^T Q
                umma_bf16_ts_w(tDK, tDP + packed_col(kk), mnmajor_desc(sQ, kk), kIdescTS,
                               (t > 0 || kk > 0) ? 1u : 0u);
            // Both slots of tile cur are free once these MMAs are done: the
            // softmax warps finished with the dO slot's lse and D before
            // signalling DS_FULL.
            umma_commit_w(&bar[BAR_Q_EMPTY + cur % kQSlots]);
            umma_commit_w(&bar[BAR_DO_EMPTY + cur % kDSlots]);
            if (t + 1 < T) {
                if (!issue_dp(cur + 1)) return false;
                if (t + 2 == T) umma_commit_w(&bar[BAR_V_EMPTY]);
            }
        }
        umma_commit_w(&bar[BAR_ACC_FULL]);
        ++acc_cnt;
        g += T;
    }
    return true;
}

__device__ bool softmax_role(const BwdParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                             uint32_t tmem, volatile int* abort_flag, int wq, int hf, int lane) {
    const int r = wq * 32 + lane;   // key row of the block = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = lane_base + 64 * hf, tDP = lane_base + 128 + 64 * hf;
    const int c0 = 64 * hf;
    const float sl = p.scale_log2;
    uint32_t g = 0, acc_cnt = 0;

    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, &bar[BAR_SCHED_FULL], &bar[BAR_SCHED_EMPTY], sched, k, abort_flag, idx))
            return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        const int j = pl.k0 + r;   // this thread's key
        const int R = p.routed_count[pl.b];
        for (int u = 0; u < pl.ntiles; ++u) {
            const uint32_t cur = g + u, st = cur % kDSlots;
            const Tile t = tile_of(pl, u);
            if (!mbar_wait_w(&bar[BAR_DO_FULL + st], (cur / kDSlots) & 1u, abort_flag, p.err))
                return false;
            const float* sL = reinterpret_cast<const float*>(smem + kOffL + st * kRowBytes) + c0;
            const float* sD = reinterpret_cast<const float*>(smem + kOffD + st * kRowBytes) + c0;
            // Visible columns [a, e] of this key: band tiles hold rows
            // row0 + c, which see j when i-W+1 <= j <= i (and i < N); far
            // tiles hold compacted routed rows, which see j when j <= i-W.
            int a, e;
            if (!t.far) {
                a = j - t.row0;
                e = min(j - t.row0 + p.W - 1, p.N - 1 - t.row0);
            } else {
                // Compacted rows ascend; the columns that see key j are those
                // with row >= j + W among the nvalid real ones.  A tile whose
                // first row is at least (last key of the block) + W is wholly
                // visible; otherwise every thread counts the rows below its
                // target, the tile's 128 row indices spread 4 per lane.
                const int* gR = p.rowidx + (size_t)pl.b * p.Npad + t.row0;
                const int nvalid = min(kBM, R + far_front(R) - t.row0);
                e = nvalid - 1;
                if (nvalid == kBM && gR[0] >= pl.k0 + kBN - 1 + p.W) {
                    a = 0;
                } else {
                    const int4 v4 = reinterpret_cast<const int4*>(gR)[lane];
                    const int cb = 4 * lane;
                    const int v0 = cb + 0 < nvalid ? v4.x : INT_MAX;
                    const int v1 = cb + 1 < nvalid ? v4.y : INT_MAX;
                    const int v2 = cb + 2 < nvalid ? v4.z : INT_MAX;
                    const int v3 = cb + 3 < nvalid ? v4.w : INT_MAX;
                    const int target = j + p.W;
                    int cnt = 0;
#pragma unroll 4
                    for (int src = 0; src < 32; ++src) {
                        cnt += __shfl_sync(0xffffffffu, v0, src) < target;
                        cnt += __shfl_sync(0xffffffffu, v1, src) < target;
                        cnt += __shfl_sync(0xffffffffu, v2, src) < target;
                        cnt += __shfl_sync(0xffffffffu, v3, src) < target;
                    }
                    a = cnt;
                }
            }
            const bool full = __all_sync(0xffffffffu, a <= c0 && e >= c0 + 63);

            // ---- phase 1: P^T
            if (!mbar_wait_w(&bar[BAR_S_FULL], cur & 1u, abort_flag, p.err)) return false;
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld32(tS, sr);
            tmem_ld32(tS + 32, sr + 32);
            tmem_ld_wait();
            float* x = reinterpret_cast<float*>(sr);
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(sL + c);
                const float2 a0 = ffma2(make_float2(x[c], x[c + 1]), make_float2(sl, sl),
                                        make_float2(-l4.x, -l4.y));
                const float2 a1 = ffma2(make_float2(x[c + 2], x[c + 3]), make_float2(sl, sl),
                                        make_float2(-l4.z, -l4.w));
                x[c] = a0.x;
                x[c + 1] = a0.y;
                x[c + 2] = a1.x;
                x[c + 3] = a1.y;
            }
            if (!full) mask_half(x, a, e, c0);
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                x[c] = ex2_approx(x[c]);
                x[c + 1] = ex2_approx(x[c + 1]);
                pk[c / 2] = pack_bf16x2(x[c], x[c + 1]);
            }
            tmem_st32(tS, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar[BAR_P_FULL]);

            // ---- phase 2: dS^T = P^T (dP^T - D)
            if (!mbar_wait_w(&bar[BAR_DP_FULL], cur & 1u, abort_flag, p.err)) return false;
            tc_fence_after();
            uint32_t dr[64];
            tmem_ld32(tDP, dr);
            tmem_ld32(tDP + 32, dr + 32);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
                const float4 d4 = *reinterpret_cast<const float4*>(sD + c);
                const float2 u0 = fadd2(make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])),
                                        make_float2(-d4.x, -d4.y));
                const float2 u1 = fadd2(make_float2(__uint_as_float(dr[c + 2]), __uint_as_float(dr[c + 3])),
                                        make_float2(-d4.z, -d4.w));
                pk[c / 2] = pack_bf16x2(x[c] * u0.x, x[c + 1] * u0.y);
                pk[c / 2 + 1] = pack_bf16x2(x[c + 2] * u1.x, x[c + 3] * u1.y);
            }
            tmem_st32(tDP, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar[BAR_DS_FULL]);
        }
        g += pl.ntiles;

        // ---- epilogue: dV and scale * dK rows of this key
        if (!mbar_wait_w(&bar[BAR_ACC_FULL], acc_cnt & 1u, abort_flag, p.err)) return false;
        ++acc_cnt;
        tc_fence_after();
        uint32_t vr[64];
        tmem_ld32(lane_base + 256 + c0, vr);
        tmem_ld32(lane_base + 256 + c0 + 32, vr + 32);
        tmem_ld_wait();
        const size_t row = ((size_t)pl.b * p.N + j) * p.Hkv + pl.kvh;
        if (j < p.N) store_row64(p.dv + row * kHD + c0, vr, 1.f);
        tmem_ld32(lane_base + 384 + c0, vr);
        tmem_ld32(lane_base + 384 + c0 + 32, vr + 32);
        tmem_ld_wait();
        if (j < p.N) store_row64(p.dk + row * kHD + c0, vr, p.scale);
        tc_fence_before();
        mbar_arrive(&bar[BAR_ACC_FREE]);
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) dkdv_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {   // operand tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(p.err, kDevErrLayout);
        // Exiting lets the dQ kernel launch: not before the schedule it reads.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    uint8_t* smem = smem_raw;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
    volatile int* sched = reinterpret_cast<volatile int*>(smem + kOffSched);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bar[BAR_K_FULL], 1);
        mbar_init(&bar[BAR_K_EMPTY], 1);
        mbar_init(&bar[BAR_V_FULL], 1);
        mbar_init(&bar[BAR_V_EMPTY], 1);
        for (int st = 0; st < kQSlots; ++st) {
            mbar_init(&bar[BAR_Q_FULL + st], 1);
            mbar_init(&bar[BAR_Q_EMPTY + st], 1);
        }
        for (int st = 0; st < kDSlots; ++st) {
            mbar_init(&bar[BAR_DO_FULL + st], 1);
            mbar_init(&bar[BAR_DO_EMPTY + st], 1);
        }
        mbar_init(&bar[BAR_S_FULL], 1);
        mbar_init(&bar[BAR_DP_FULL], 1);
        mbar_init(&bar[BAR_P_FULL], kSoftmaxThreads);
        mbar_init(&bar[BAR_DS_FULL], kSoftmaxThreads);
        mbar_init(&bar[BAR_ACC_FULL], 1);
        mbar_init(&bar[BAR_ACC_FREE], kSoftmaxThreads);
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
    // Launched as a programmatic dependent of the backward schedule: the
    // prologue above overlaps it, and its work lists and compacted rows are
    // read only after this wait.  The dQ kernel after this one may launch
    // from here on: it reads nothing this kernel writes, and what it reads
    // is complete now.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp < 8) {
        warpgroup_reg_inc<kRegsSoftmax>();
        softmax_role(p, smem, bar, sched, tmem, abort_flag, warp & 3, warp >> 2, lane);
    } else {
        warpgroup_reg_dec<kRegsOther>();
    }
    if (warp == 8) {
        if (lane == 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_qc);
            prefetch_tensormap(&p.tm_do);
            prefetch_tensormap(&p.tm_doc);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
        }
        __syncwarp();
        KvIssued n_is{0, 0, 0, 0};
        if (!producer(p, smem, bar, sched, abort_flag, n_is)) {
            drain_ring(&bar[BAR_Q_FULL], kQSlots, n_is.q);
            drain_ring(&bar[BAR_DO_FULL], kDSlots, n_is.d);
            drain_ring(&bar[BAR_K_FULL], 1, n_is.k);
            drain_ring(&bar[BAR_V_FULL], 1, n_is.v);
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

}  // namespace kv

// ====================================================================== dQ ==
namespace dqk {

// Key tiles live from S(j) to dQ += dS(j) K(j), value tiles only until dP(j):
// three key slots and two value slots keep the loads a block and more ahead.
constexpr int kKSlots = 3;
constexpr int kVSlots = 2;
constexpr int kOffQ = 0;
constexpr int kOffDO = kOffQ + kTileBytes;
constexpr int kOffK = kOffDO + kTileBytes;              // [kKSlots] key tiles
constexpr int kOffV = kOffK + kKSlots * kTileBytes;     // [kVSlots] value tiles
constexpr int kOffBar = kOffV + kVSlots * kTileBytes;

enum {
    BAR_Q_FULL = 0,
    BAR_Q_EMPTY,
    BAR_K_FULL,                            // [kKSlots]
    BAR_K_EMPTY = BAR_K_FULL + kKSlots,    // [kKSlots]
    BAR_V_FULL = BAR_K_EMPTY + kKSlots,    // [kVSlots]
    BAR_V_EMPTY = BAR_V_FULL + kVSlots,    // [kVSlots]
    BAR_S_FULL = BAR_V_EMPTY + kVSlots,    // [2] one per S buffer
    BAR_DP_FULL = BAR_S_FULL + 2,
    BAR_DS_FULL,
    BAR_ACC_FULL,
    BAR_ACC_FREE,
    BAR_SCHED_FULL,
    BAR_SCHED_EMPTY = BAR_SCHED_FULL + kSched,
    BAR_DRAIN = BAR_SCHED_EMPTY + kSched,
    BAR_COUNT
};
constexpr int kOffSched = kOffBar + BAR_COUNT * 8;
constexpr int kOffMisc = kOffSched + kSched * 4;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Plan {
    int b, h, kvh, row0, kv0, nblk;
    bool far;
};

__device__ __forceinline__ Plan make_plan(const BwdParams& p, int idx) {
    const BwdItem it = load_item(p, idx);
    Plan pl;
    pl.b = it.b;
    pl.h = it.h;
    pl.kvh = it.h / (p.Hq / p.Hkv);
    pl.far = it.kind == kBwdQFar;
    pl.row0 = it.t * kBM;
    pl.kv0 = it.a0;
    pl.nblk = it.a1;
    return pl;
}

// Loads issued so far on each ring of the dQ producer (see KvIssued).
struct QIssued {
    uint32_t q, k, v;
};

__device__ bool producer(const BwdParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                         volatile int* abort_flag, QIssued& n_is) {
    const int n = p.n_items[0];
    for (int k = 0;; ++k) {
        int idx;
        if (!publish_item(p, &bar[BAR_SCHED_FULL], &bar[BAR_SCHED_EMPTY], sched, k, n,
                          abort_flag, idx))
            return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        if (!mbar_wait_w(&bar[BAR_Q_EMPTY], (n_is.q & 1u) ^ 1u, abort_flag, p.err)) return false;
        mbar_arrive_expect_tx_w(&bar[BAR_Q_FULL], 2 * kTileBytes);
        load_tile_pair(pl.far ? &p.tm_qc : &p.tm_q, smem + kOffQ, &bar[BAR_Q_FULL], pl.h, pl.row0,
                       pl.b);
        load_tile_pair(pl.far ? &p.tm_doc : &p.tm_do, smem + kOffDO, &bar[BAR_Q_FULL], pl.h,
                       pl.row0, pl.b);
        ++n_is.q;
        for (int j = 0; j < pl.nblk; ++j) {
            const int key0 = pl.kv0 + j * kBN;
            const uint32_t ks = n_is.k % kKSlots, kph = (n_is.k / kKSlots) & 1u;
            if (!mbar_wait_w(&bar[BAR_K_EMPTY + ks], kph ^ 1u, abort_flag, p.err)) return false;
            mbar_arrive_expect_tx_w(&bar[BAR_K_FULL + ks], kTileBytes);
            load_tile_pair(&p.tm_k, smem + kOffK + ks * kTileBytes, &bar[BAR_K_FULL + ks], pl.kvh,
                           key0, pl.b);
            ++n_is.k;
            const uint32_t vs = n_is.v % kVSlots, vph = (n_is.v / kVSlots) & 1u;
            if (!mbar_wait_w(&bar[BAR_V_EMPTY + vs], vph ^ 1u, abort_flag, p.err)) return false;
            mbar_arrive_expect_tx_w(&bar[BAR_V_FULL + vs], kTileBytes);
            load_tile_pair(&p.tm_v, smem + kOffV + vs * kTileBytes, &bar[BAR_V_FULL + vs], pl.kvh,
                           key0, pl.b);
            ++n_is.v;
        }
    }
    return true;
}

__device__ bool mma_issuer(const BwdParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                           uint32_t tmem, volatile int* abort_flag) {
    const uint32_t tDP = tmem + 256, tDQ = tmem + 384;
    const uint32_t sQ = smem_u32(smem + kOffQ), sDO = smem_u32(smem + kOffDO);
    uint32_t g = 0, q_cnt = 0, acc_cnt = 0;

    // Block c (a running count over items): key slot c % kKSlots, value slot
    // c % kVSlots, S buffer c % 2.
    auto issue_s = [&](uint32_t c) -> bool {   // S = Q K^T
        const uint32_t ks = c % kKSlots, buf = c % 2;
        if (!mbar_wait_w(&bar[BAR_K_FULL + ks], (c / kKSlots) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + kOffK + ks * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk)
            umma_bf16_w(tmem + 128 * buf, kmajor_desc(sQ, kk), kmajor_desc(sK, kk), kIdescSS,
                        kk > 0 ? 1u : 0u);
        umma_commit_w(&bar[BAR_S_FULL + buf]);
        return true;
    };
    auto issue_dp = [&](uint32_t c) -> bool {   // dP = dO V^T, then the value slot is free
        const uint32_t vs = c % kVSlots;
        if (!mbar_wait_w(&bar[BAR_V_FULL + vs], (c / kVSlots) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + kOffV + vs * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk)
            umma_bf16_w(tDP, kmajor_desc(sDO, kk), kmajor_desc(sV, kk), kIdescSS, kk > 0 ? 1u : 0u);
        umma_commit_w(&bar[BAR_DP_FULL]);
        umma_commit_w(&bar[BAR_V_EMPTY + vs]);
        return true;
    };

    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, &bar[BAR_SCHED_FULL], &bar[BAR_SCHED_EMPTY], sched, k, abort_flag, idx))
            return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        const int n = pl.nblk;
        if (!mbar_wait_w(&bar[BAR_Q_FULL], q_cnt & 1u, abort_flag, p.err)) return false;
        ++q_cnt;
        if (!issue_s(g) || !issue_dp(g)) return false;
        for (int j = 0; j < n; ++j) {
            const uint32_t cur = g + j;
            if (j + 1 < n && !issue_s(cur + 1)) return false;
            if (!mbar_wait_w(&bar[BAR_DS_FULL], cur & 1u, abort_flag, p.err)) return false;
            if (j == 0 && !mbar_wait_w(&bar[BAR_ACC_FREE], (acc_cnt & 1u) ^ 1u, abort_flag, p.err))
                return false;
            tc_fence_after();
            if (j + 1 < n && !issue_dp(cur + 1)) return false;
            const uint32_t ks = cur % kKSlots;
            const uint32_t sK = smem_u32(smem + kOffK + ks * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)   // dQ += dS K
                umma_bf16_ts_w(tDQ, tmem + 128 * (cur % 2) + packed_col(kk), mnmajor_desc(sK, kk),
                               kIdescTS, (j > 0 || kk > 0) ? 1u : 0u);
            umma_commit_w(&bar[BAR_K_EMPTY + ks]);
        }
        umma_commit_w(&bar[BAR_ACC_FULL]);
        umma_commit_w(&bar[BAR_Q_EMPTY]);
        ++acc_cnt;
        g += n;
    }
    return true;
}

__device__ bool softmax_role(const BwdParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                             uint32_t tmem, volatile int* abort_flag, int wq, int hf, int lane) {
    const int r = wq * 32 + lane;   // query row of the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const int c0 = 64 * hf;
    const float sl = p.scale_log2;
    uint32_t g = 0, acc_cnt = 0;

    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, &bar[BAR_SCHED_FULL], &bar[BAR_SCHED_EMPTY], sched, k, abort_flag, idx))
            return false;
        if (idx < 0) break;
        const Plan pl = make_plan(p, idx);
        int i = -1;
        if (pl.far) {
            const int v = p.rowidx[(size_t)pl.b * p.Npad + pl.row0 + r];
            i = v >= 0 ? v : -1;
        } else if (pl.row0 + r < p.N) {
            i = pl.row0 + r;
        }
        const size_t stat = ((size_t)pl.b * p.Hq + pl.h) * p.Npad + pl.row0 + r;
        const float lrow = (pl.far ? p.l_far : p.l_band)[stat];
        const float drow = (pl.far ? p.d_far : p.d_band)[stat];
        const float2 sl2 = make_float2(sl, sl), nl2 = make_float2(-lrow, -lrow);
        const float2 nd2 = make_float2(-drow, -drow);
        for (int j = 0; j < pl.nblk; ++j) {
            const uint32_t cur = g + j, buf = cur % 2;
            const int key0 = pl.kv0 + j * kBN;
            // Visible keys of row i, as block columns [a, e]: window rows
            // [i-W+1, i], far rows [0, i]; no row: empty.
            int a = 1, e = 0;
            if (i >= 0) {
                a = pl.far ? 0 : i - p.W + 1 - key0;
                e = i - key0;
            }
            const bool full = __all_sync(0xffffffffu, a <= c0 && e >= c0 + 63);
            if (!mbar_wait_w(&bar[BAR_S_FULL + buf], (cur / 2) & 1u, abort_flag, p.err)) return false;
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld32(lane_base + 128 * buf + c0, sr);
            tmem_ld32(lane_base + 128 * buf + c0 + 32, sr + 32);
            tmem_ld_wait();
            float* x = reinterpret_cast<float*>(sr);
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const float2 y = ffma2(make_float2(x[c], x[c + 1]), sl2, nl2);
                x[c] = y.x;
                x[c + 1] = y.y;
            }
            if (!full) mask_half(x, a, e, c0);
#pragma unroll
            for (int c = 0; c < 64; ++c) x[c] = ex2_approx(x[c]);
            if (!mbar_wait_w(&bar[BAR_DP_FULL], cur & 1u, abort_flag, p.err)) return false;
            tc_fence_after();
            uint32_t dr[64];
            tmem_ld32(lane_base + 256 + c0, dr);
            tmem_ld32(lane_base + 256 + c0 + 32, dr + 32);
            tmem_ld_wait();
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const float2 u = fadd2(make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), nd2);
                pk[c / 2] = pack_bf16x2(x[c] * u.x, x[c + 1] * u.y);
            }
            tmem_st32(lane_base + 128 * buf + c0, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar[BAR_DS_FULL]);
        }
        g += pl.nblk;

        // ---- epilogue: scale * dQ of this row (band tiles skip far rows)
        if (!mbar_wait_w(&bar[BAR_ACC_FULL], acc_cnt & 1u, abort_flag, p.err)) return false;
        ++acc_cnt;
        tc_fence_after();
        uint32_t qr[64];
        tmem_ld32(lane_base + 384 + c0, qr);
        tmem_ld32(lane_base + 384 + c0 + 32, qr + 32);
        tmem_ld_wait();
        bool write = i >= 0;
        if (write && !pl.far) write = !(p.gate[(size_t)pl.b * p.N + i] != 0 && i >= p.W);
        if (write)
            store_row64(p.dq + (((size_t)pl.b * p.N + i) * p.Hq + pl.h) * kHD + c0, qr, p.scale);
        tc_fence_before();
        mbar_arrive(&bar[BAR_ACC_FREE]);
    }
    return true;
}

__global__ void __launch_bounds__(kThreads, 1) dq_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
    volatile int* sched = reinterpret_cast<volatile int*>(smem + kOffSched);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bar[BAR_Q_FULL], 1);
        mbar_init(&bar[BAR_Q_EMPTY], 1);
        for (int st = 0; st < kKSlots; ++st) {
            mbar_init(&bar[BAR_K_FULL + st], 1);
            mbar_init(&bar[BAR_K_EMPTY + st], 1);
        }
        for (int st = 0; st < kVSlots; ++st) {
            mbar_init(&bar[BAR_V_FULL + st], 1);
            mbar_init(&bar[BAR_V_EMPTY + st], 1);
        }
        for (int st = 0; st < 2; ++st) mbar_init(&bar[BAR_S_FULL + st], 1);
        mbar_init(&bar[BAR_DP_FULL], 1);
        mbar_init(&bar[BAR_DS_FULL], kSoftmaxThreads);
        mbar_init(&bar[BAR_ACC_FULL], 1);
        mbar_init(&bar[BAR_ACC_FREE], kSoftmaxThreads);
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
        softmax_role(p, smem, bar, sched, tmem, abort_flag, warp & 3, warp >> 2, lane);
    } else {
        warpgroup_reg_dec<kRegsOther>();
    }
    if (warp == 8) {
        if (lane == 0) {
            prefetch_tensormap(&p.tm_q);
            prefetch_tensormap(&p.tm_qc);
            prefetch_tensormap(&p.tm_do);
            prefetch_tensormap(&p.tm_doc);
            prefetch_tensormap(&p.tm_k);
            prefetch_tensormap(&p.tm_v);
        }
        __syncwarp();
        QIssued n_is{0, 0, 0};
        if (!producer(p, smem, bar, sched, abort_flag, n_is)) {
            drain_ring(&bar[BAR_K_FULL], kKSlots, n_is.k);
            drain_ring(&bar[BAR_V_FULL], kVSlots, n_is.v);
            drain_ring(&bar[BAR_Q_FULL], 1, n_is.q);
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

}  // namespace dqk

bool fill_params(BwdParams& p, const TcBwdArgs& a, unsigned int* err) {
    memset(&p, 0, sizeof(p));
    const BwdWs& L = *a.L;
    const uint64_t N = a.N, B = a.B, Np = L.Npad;
    bool ok = make_tmap_4d_bf16(&p.tm_q, a.q, kHD, a.Hq, N, B, 64, kBM) &&
              make_tmap_4d_bf16(&p.tm_qc, a.ws + L.qc, kHD, a.Hq, Np, B, 64, kBM) &&
              make_tmap_4d_bf16(&p.tm_do, a.d_o, kHD, a.Hq, N, B, 64, kBM) &&
              make_tmap_4d_bf16(&p.tm_doc, a.ws + L.doc, kHD, a.Hq, Np, B, 64, kBM) &&
              make_tmap_4d_bf16(&p.tm_k, a.k, kHD, a.Hkv, N, B, 64, kBN) &&
              make_tmap_4d_bf16(&p.tm_v, a.v, kHD, a.Hkv, N, B, 64, kBN);
    if (!ok) return false;
    p.routed_count = reinterpret_cast<const int*>(a.ws + L.routed_count);
    p.rowidx = reinterpret_cast<const int*>(a.ws + L.rowidx);
    p.d_band = reinterpret_cast<const float*>(a.ws + L.d_band);
    p.l_band = reinterpret_cast<const float*>(a.ws + L.l_band);
    p.d_far = reinterpret_cast<const float*>(a.ws + L.d_far);
    p.l_far = reinterpret_cast<const float*>(a.ws + L.l_far);
    p.gate = a.gate;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.err = err;
    p.B = a.B;
    p.N = a.N;
    p.Npad = L.Npad;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.W = a.W;
    p.scale = a.scale;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    return true;
}

}  // namespace

cudaError_t launch_bwd_dkdv(const TcBwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
    BwdParams p;
    if (!fill_params(p, a, err)) return cudaErrorInvalidValue;
    int* counters = reinterpret_cast<int*>(a.ws + a.L->counters);
    p.items = reinterpret_cast<const BwdItem*>(a.ws + a.L->items_kv);
    p.n_items = counters;
    p.next_item = counters + 1;
    static std::atomic<uint64_t> smem_allowed{0};
    cudaError_t e = allow_dynamic_smem(kv::dkdv_kernel, kv::kSmemBytes, smem_allowed);
    if (e != cudaSuccess) return e;
    // A programmatic dependent launch of the backward schedule before it on
    // the stream (the kernel waits for that grid before reading its lists).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kv::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kv::dkdv_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const TcBwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s) {
    BwdParams p;
    if (!fill_params(p, a, err)) return cudaErrorInvalidValue;
    int* counters = reinterpret_cast<int*>(a.ws + a.L->counters);
    p.items = reinterpret_cast<const BwdItem*>(a.ws + a.L->items_q);
    p.n_items = counters + 2;
    p.next_item = counters + 3;
    static std::atomic<uint64_t> smem_allowed{0};
    cudaError_t e = allow_dynamic_smem(dqk::dq_kernel, dqk::kSmemBytes, smem_allowed);
    if (e != cudaSuccess) return e;
    // Launched as a programmatic dependent of the dK/dV kernel before it on
    // the stream: the two read the same inputs and write disjoint outputs, so
    // dQ CTAs start on the SMs the dK/dV kernel's last items leave idle.  Its
    // own inputs (work list, compacted rows) are complete before any dK/dV
    // CTA lets it launch.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dqk::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, dqk::dq_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t bwd_set_wait_limit(uint64_t ns) { return set_wait_limit_of_unit(ns); }

}  // namespace swi
