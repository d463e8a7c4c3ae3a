// Routed prefill on the 5th-generation tensor cores (sm_103a): two query
// tiles per CTA sharing every K/V block.
//
// A work item holds 256 query rows of one (batch, head): two 128-row tiles A
// and B.  Band items take 256 consecutive rows and walk their window keys; far
// items take 256 compacted routed rows and walk keys [0, max i] (a far item
// may hold one of its two tiles alone, the other then inactive).  The CTA
// streams one sequence of 64-key blocks; each tile uses the contiguous run of
// blocks its rows can see, so every K/V block is loaded once for both tiles.
//
// Items are claimed dynamically from the cost-sorted list (longest first).
//
// Per tile and block: S = Q K^T (TMEM) -> softmax (P, bf16, written back over
// S in TMEM) -> O += P V (P read from TMEM).  Each tile has two S buffers, so
// the tensor core computes S of block j+1 while the softmax warps work on
// block j: per step the MMA warp issues S(j+1) of both tiles, then PV(j) of
// both tiles as their P become ready.  A tile's softmax thus has a whole step
// of tensor work (both tiles' PV and next S) to finish in, and the tensor core
// does not wait on the softmax in steady state.
//   warps 0-3   softmax + epilogue of tile A (thread r owns row r = TMEM lane r)
//               (the epilogue stages rows in shared memory for coalesced stores)
//   warps 4-7   softmax + epilogue of tile B
//   warp 8      item claimer and TMA producer: Q tiles of band items, K and V
//               blocks (converged, elected issue)
//   warp 9      TMEM allocator and MMA issuer of tile A (converged, elected issue)
//   warp 10     Q of far items: gathers the tile's routed rows by row index
//               straight from Q (cp.async into the swizzled tile layout)
//   warp 11     MMA issuer of tile B
// TMEM: S_A0 [0,64), S_A1 [64,128), S_B0 [128,192), S_B1 [192,256),
// O_A [256,384), O_B [384,512).
// Key sets per row (SwiAttn report, section 2; window per the weimeta.cn SWA
// glossary): window rows [max(0, i-W+1), i], routed rows [0, i].  With S
// global anchors (the glossary's 全局锚点) window rows also see
// [0, min(S, i-W+1)): a band item then starts with an anchor run of blocks
// from key 0 before its window run.

#include "ptx.cuh"
#include "swiattn_internal.h"

#include <cuda_bf16.h>
#include <math.h>

namespace swi {
namespace {

constexpr int kKB = 64;      // keys per block
constexpr int kStages = 4;
constexpr int kThreads = 384;   // 3 warpgroups
// Launched at 168 registers per thread (12 warps x 32 x 168 = 64512); the
// producer/MMA warpgroup gives up registers to the two softmax warpgroups:
// 2 x 128 x 216 + 128 x 72 = 64512.
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsOther = 72;
constexpr int kTileBytes = kBM * kHD * 2;    // 32 KiB: one Q tile
constexpr int kHalfBytes = kTileBytes / 2;   // 16 KiB: 64 head-dim columns of it
constexpr int kKVBytes = kKB * kHD * 2;      // 16 KiB: one K or V block
constexpr int kKVHalf = kKVBytes / 2;        // 8 KiB

constexpr int kSched = 4;                                 // item broadcast ring
constexpr int kStageBytesPerWarp = 32 * 64 * 2;           // 32 rows x 64 bf16 output columns

constexpr int kOffQ = 0;                                  // Q_A, Q_B
constexpr int kOffK = kOffQ + 2 * kTileBytes;             // K slots
constexpr int kOffV = kOffK + kStages * kKVBytes;         // V slots
constexpr int kOffStage = kOffV + kStages * kKVBytes;     // epilogue staging, 8 warps
constexpr int kOffBar = kOffStage + 8 * kStageBytesPerWarp;

enum {
    BAR_Q_FULL = 0,                        // [2] per tile
    BAR_Q_EMPTY = BAR_Q_FULL + 2,          // [2]
    BAR_KV_FULL = BAR_Q_EMPTY + 2,         // [kStages]: slot of step g holds K_j and V_{j-1}
    BAR_KV_EMPTY = BAR_KV_FULL + kStages,  // [kStages]
    BAR_S_FULL = BAR_KV_EMPTY + kStages,   // [4]: tile x, S buffer b at 2x + b
    BAR_P_FULL = BAR_S_FULL + 4,           // [4]
    BAR_O_DONE = BAR_P_FULL + 4,           // [2]: a PV other than the run's last completed
    BAR_O_FULL = BAR_O_DONE + 2,           // [2]: the run's last PV completed
    BAR_O_FREE = BAR_O_FULL + 2,           // [2]
    BAR_SCHED_FULL = BAR_O_FREE + 2,       // [kSched]
    BAR_SCHED_EMPTY = BAR_SCHED_FULL + kSched,
    BAR_DRAIN = BAR_SCHED_EMPTY + kSched,
    BAR_COUNT
};
// Consumers of a broadcast item: the two MMA warps, the eight softmax warps
// and the far-query gatherer.
constexpr uint32_t kSchedConsumers = 2 + 8 + 1;

constexpr int kOffSched = kOffBar + BAR_COUNT * 8;
constexpr int kOffMisc = kOffSched + kSched * 4;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t col_s(int x, uint32_t b) { return x * 128u + b * 64u; }
__device__ __forceinline__ uint32_t col_o(int x) { return x ? 384u : 256u; }

constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kKB, false, false);
constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, kHD, false, true);

struct PfParams {
    CUtensorMap tm_q, tm_k, tm_v;
    const __nv_bfloat16* q;  // [B, N, Hq, 128]: far tiles gather their rows from it
    const int* routed_list;
    const int* routed_count;
    const int* tile_prefix;
    const int* n_items;
    int* next_item;          // work counter, zeroed by the schedule
    const WorkItem* items;
    const uint8_t* gate;
    __nv_bfloat16* o;
    float* lse;
    unsigned int* err;
    int B, N, Hq, Hkv, W, NT;
    int S;             // global anchors of window rows (0: none)
    float scale_log2;
};

struct Plan {
    int b, h, kvh, kind;
    int row0;          // band: first query row of tile A; far: first compacted index of tile A
    int kv0, nblk;     // first key of the window run and the block sequence's length
    int na;            // anchor blocks at the head of the sequence (keys from 0)
    int ja1[2];        // anchor run per tile: blocks 0 .. ja1 (-1: none)
    int j0[2], j1[2];  // window (or far) run per tile (j0 > j1: tile empty)
    int rlo[2], nrows[2];   // valid local rows of each tile: [rlo, nrows)
};

template <bool ANCH>
__device__ __forceinline__ Plan make_plan(const PfParams& p, int idx) {
    const WorkItem it = p.items[idx];
    Plan pl;
    pl.b = it.b;
    pl.h = it.h;
    pl.kvh = it.h / (p.Hq / p.Hkv);
    pl.kind = it.kind;
    pl.row0 = it.tile * 2 * kBM;
    pl.rlo[0] = pl.rlo[1] = 0;
    pl.na = 0;
    pl.ja1[0] = pl.ja1[1] = -1;
    if (it.kind != kItemBand) {   // a far pair, or one of its tiles alone
        const int cnt = p.routed_count[it.b];
        const int* list = p.routed_list + (size_t)it.b * p.N;
        // The first far tile holds the count's remainder (its first `front`
        // slots are empty), so the part-filled tile walks the shortest key
        // range, not the longest.  Local row r of tile x is compacted row
        // row0 + 128 x + r.
        pl.row0 -= far_front(cnt);
        pl.kv0 = 0;
        int maxb = 0;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int r0 = pl.row0 + x * kBM;
            const bool off = it.kind == (x == 0 ? kItemFarB : kItemFarA);
            pl.rlo[x] = max(0, -r0);
            pl.nrows[x] = off ? 0 : max(0, min(kBM, cnt - r0));
            pl.j0[x] = 0;
            pl.j1[x] = pl.nrows[x] > pl.rlo[x] ? list[r0 + pl.nrows[x] - 1] / kKB : -1;
            maxb = max(maxb, pl.j1[x] + 1);
        }
        pl.nblk = maxb;
    } else {
        const int q0 = pl.row0;
        pl.kv0 = max(0, q0 - p.W + 1);
        const int* pre = p.tile_prefix + (size_t)it.b * (p.NT + 1);
        int last = -1;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int r0 = q0 + x * kBM;
            pl.nrows[x] = max(0, min(kBM, p.N - r0));
            const int t = r0 / kBM;
            const bool has_rows = pl.nrows[x] > 0 && (pre[t + 1] - pre[t]) < pl.nrows[x];
            if (has_rows) {
                const int lo_key = max(0, r0 - p.W + 1);
                const int hi_key = r0 + pl.nrows[x] - 1;
                pl.j0[x] = (lo_key - pl.kv0) / kKB;
                pl.j1[x] = (hi_key - pl.kv0) / kKB;
                last = max(last, pl.j1[x]);
                const int hi_anchor = min(p.S - 1, hi_key - p.W);   // anchors below the window
                if (ANCH && hi_anchor >= 0) {
                    pl.ja1[x] = hi_anchor / kKB;
                    pl.na = max(pl.na, pl.ja1[x] + 1);
                }
            } else {
                pl.j0[x] = 1;
                pl.j1[x] = 0;
            }
        }
        // The window runs follow the anchor blocks.
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            pl.j0[x] += pl.na;
            pl.j1[x] += pl.na;
        }
        pl.nblk = last + 1 + pl.na;
    }
    return pl;
}

__device__ __forceinline__ bool tile_active(const Plan& pl, int x) { return pl.j0[x] <= pl.j1[x]; }
template <bool ANCH>
__device__ __forceinline__ bool blk_active(const Plan& pl, int x, int j) {
    return (ANCH && j <= pl.ja1[x]) || (j >= pl.j0[x] && j <= pl.j1[x]);
}
template <bool ANCH>
__device__ __forceinline__ int first_blk(const Plan& pl, int x) {
    return (ANCH && pl.ja1[x] >= 0) ? 0 : pl.j0[x];
}
template <bool ANCH>
__device__ __forceinline__ int blk_key0(const Plan& pl, int j) {
    return (ANCH && j < pl.na) ? j * kKB : pl.kv0 + (j - (ANCH ? pl.na : 0)) * kKB;
}

// ----------------------------------------------------------------- roles --
//
// Items are taken dynamically, longest first (the list is cost-sorted): the
// producer warp claims the next index with an atomic and broadcasts it through
// a kSched-slot ring in shared memory; a negative index ends the stream.

// Producer side: claim item k's index and publish it (or -1 past the end).
__device__ bool publish_item(const PfParams& p, uint64_t* bar, volatile int* sched, int k, int n,
                             volatile int* abort_flag, int& idx) {
    const int slot = k % kSched;
    const uint32_t par = (static_cast<uint32_t>(k) / kSched) & 1u;
    if (!mbar_wait_w(&bar[BAR_SCHED_EMPTY + slot], par ^ 1u, abort_flag, p.err)) return false;
    int v = 0;
    if ((threadIdx.x & 31) == 0) v = atomicAdd(p.next_item, 1);
    v = __shfl_sync(0xffffffffu, v, 0);
    idx = v < n ? v : -1;
    if ((threadIdx.x & 31) == 0) {
        sched[slot] = idx;
        mbar_arrive(&bar[BAR_SCHED_FULL + slot]);   // release: the write above is visible
    }
    __syncwarp();
    return true;
}

// Consumer side (a whole warp): read item k's index and free its slot.
__device__ bool consume_item(const PfParams& p, uint64_t* bar, volatile int* sched, int k,
                             volatile int* abort_flag, int& idx) {
    const int slot = k % kSched;
    const uint32_t par = (static_cast<uint32_t>(k) / kSched) & 1u;
    if (!mbar_wait_w(&bar[BAR_SCHED_FULL + slot], par, abort_flag, p.err)) return false;
    idx = sched[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&bar[BAR_SCHED_EMPTY + slot]);
    return true;
}

// Producer warp (converged, one elected lane issues): per item, the Q tiles,
// then one K/V slot per step g: step j of an item carries K_j (j < nblk) and
// V_{j-1} (j >= 1), so a slot is freed by one commit after S(j) and PV(j-1).
//
// Each Q slot sees one load per active tile per item, band (TMA, here) or far
// (the gatherer warp).  This warp waits for the slot of every load, in order;
// it finishes an item's waits before it publishes the next item, and the slot
// is freed again only after the tile's last S, which needs this warp's K/V
// loads, issued after its wait: so each wait finds the barrier at the phase
// it names or the one before.  The gatherer's waits (far loads only) are
// argued at q_gatherer.
template <bool ANCH>
__device__ bool producer(const PfParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                         volatile int* abort_flag, uint32_t& g, uint32_t* q_issued, bool* q_tma_last) {
    const int n = *p.n_items;
    for (int k = 0;; ++k) {
        int idx;
        if (!publish_item(p, bar, sched, k, n, abort_flag, idx)) return false;
        if (idx < 0) break;
        const Plan pl = make_plan<ANCH>(p, idx);
        const bool far = pl.kind != kItemBand;
        auto load_q = [&](int x) -> bool {
            if (!mbar_wait_w(&bar[BAR_Q_EMPTY + x], (q_issued[x] & 1u) ^ 1u, abort_flag, p.err)) return false;
            ++q_issued[x];
            q_tma_last[x] = !far;
            if (far) return true;
            mbar_arrive_expect_tx_w(&bar[BAR_Q_FULL + x], kTileBytes);
            uint8_t* dst = smem + kOffQ + x * kTileBytes;
            const int row = pl.row0 + x * kBM;
            tma_load_4d_w(dst, &p.tm_q, &bar[BAR_Q_FULL + x], 0, pl.h, row, pl.b);
            tma_load_4d_w(dst + kHalfBytes, &p.tm_q, &bar[BAR_Q_FULL + x], 64, pl.h, row, pl.b);
            return true;
        };
        if (tile_active(pl, 0) && !load_q(0)) return false;
        for (int j = 0; j <= pl.nblk; ++j) {
            if (j < pl.nblk && tile_active(pl, 1) && j == first_blk<ANCH>(pl, 1) && !load_q(1)) return false;
            const uint32_t st = g % kStages, ph = (g / kStages) & 1u;
            if (!mbar_wait_w(&bar[BAR_KV_EMPTY + st], ph ^ 1u, abort_flag, p.err)) return false;
            const uint32_t bytes = (j < pl.nblk ? kKVBytes : 0) + (j >= 1 ? kKVBytes : 0);
            mbar_arrive_expect_tx_w(&bar[BAR_KV_FULL + st], bytes);
            if (j < pl.nblk) {
                uint8_t* dst = smem + kOffK + st * kKVBytes;
                const int key0 = blk_key0<ANCH>(pl, j);
                tma_load_4d_w(dst, &p.tm_k, &bar[BAR_KV_FULL + st], 0, pl.kvh, key0, pl.b);
                tma_load_4d_w(dst + kKVHalf, &p.tm_k, &bar[BAR_KV_FULL + st], 64, pl.kvh, key0, pl.b);
            }
            if (j >= 1) {
                uint8_t* dst = smem + kOffV + st * kKVBytes;
                const int key0 = blk_key0<ANCH>(pl, j - 1);
                tma_load_4d_w(dst, &p.tm_v, &bar[BAR_KV_FULL + st], 0, pl.kvh, key0, pl.b);
                tma_load_4d_w(dst + kKVHalf, &p.tm_v, &bar[BAR_KV_FULL + st], 64, pl.kvh, key0, pl.b);
            }
            ++g;
        }
    }
    return true;
}

// Far-query gatherer (warp 10).  Row r of far tile x is compacted routed row
// c = row0 + 128x + r, i.e. query row routed_list[c]; its 256 bytes (head h)
// are copied in 16-byte chunks with cp.async into the same 128-byte-swizzled
// K-major layout the TMA writes for band tiles: chunk u of the row (half u/8)
// lands at 16-byte slot (u%8) ^ (r%8) of the row's 128 bytes.  Rows outside
// [0, routed count) (the first far tile's empty front slots, rows past the
// count) are zero-filled.  Half-warps take one row each, so every load
// instruction reads two whole rows.  The copies complete, each lane fences its
// writes for the tensor core's async proxy, then one arrival fills the slot.
__device__ void gather_far_q(const PfParams& p, uint8_t* smem, uint64_t* bar, const Plan& pl, int x,
                             int lane) {
    const int R = p.routed_count[pl.b];
    const int c0 = pl.row0 + x * kBM;
    const int* list = p.routed_list + (size_t)pl.b * p.N;
    int src[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        src[u] = (c >= 0 && c < R) ? list[c] : -1;
    }
    const uint32_t tile = smem_u32(smem + kOffQ + x * kTileBytes);
    const int sub = lane & 15;
    const uint32_t col = (sub >> 3) * kHalfBytes;
    const uint32_t slot = sub & 7;
    const size_t head = (size_t)pl.b * p.N * p.Hq + pl.h;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {   // rows 32 q4 .. 32 q4 + 31; lane l holds row 32 q4 + l's index
#pragma unroll 4
        for (int it = q4 * 16; it < q4 * 16 + 16; ++it) {
            const int r = 2 * it + (lane >> 4);
            const int i = __shfl_sync(0xffffffffu, src[q4], r & 31);
            const uint32_t dst = tile + col + r * 128 + ((slot ^ (r & 7)) << 4);
            const __nv_bfloat16* s = p.q + (head + (size_t)max(i, 0) * p.Hq) * kHD + sub * 8;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(s),
                         "r"(i >= 0 ? 16u : 0u)
                         : "memory");
        }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar[BAR_Q_FULL + x]);
    __syncwarp();
}

template <bool ANCH>
__device__ bool q_gatherer(const PfParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                           volatile int* abort_flag, int lane) {
    uint32_t cnt[2] = {0, 0};
    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, bar, sched, k, abort_flag, idx)) return false;
        if (idx < 0) break;
        const Plan pl = make_plan<ANCH>(p, idx);
        // Every load of a slot counts (cnt: its phase), but the gatherer
        // waits only before its own (far) loads.  Such a wait names the
        // previous load's release and finds the barrier at that phase or
        // just past it: not further past (the next release needs this load's
        // rows), nor further back (the producer waited for the release before
        // that one before it issued the previous load, in an earlier item,
        // and published this item only after).  Waiting before band loads as
        // well, which need nothing from this warp, could find the slot freed
        // once more already and then wait for a phase that never comes.
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            if (!tile_active(pl, x)) continue;
            const uint32_t use = cnt[x]++;
            if (pl.kind == kItemBand) continue;
            if (!mbar_wait_w(&bar[BAR_Q_EMPTY + x], (use & 1u) ^ 1u, abort_flag, p.err)) return false;
            gather_far_q(p, smem, bar, pl, x, lane);
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

// MMA warp of tile x (one per tile, converged, elected issue).  Step j of an
// item (slot g holds K_j and V_{j-1}): S(j), if the tile's run contains block
// j, into the S buffer not holding block j-1's P; then PV(j-1) once the
// softmax has written P(j-1).  A tile's S buffer is reused two blocks later,
// after the PV that read it (this warp issues both, in that order).  Each PV
// but the run's last commits BAR_O_DONE (the softmax waits on it before
// rescaling O); the last commits BAR_O_FULL.  Both MMA warps walk every step
// and release the slot with one commit each; the tensor core interleaves
// their MMAs, which touch disjoint TMEM columns.
template <bool ANCH>
__device__ bool mma_issuer(const PfParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                           uint32_t tmem, volatile int* abort_flag, int x) {
    uint32_t g = 0, q_cnt = 0, s_cnt = 0, o_cnt = 0;
    // Shared-memory descriptors of the operand tiles, formed once: the start
    // address is the low field, so a byte offset o within a tile adds o >> 4
    // (no carry: every address in the 227 KiB window is below 2^18).
    const uint64_t dQ = sdesc_sw128(smem_u32(smem + kOffQ + x * kTileBytes), 16, 1024);
    const uint64_t dK0 = sdesc_sw128(smem_u32(smem + kOffK), 16, 1024);
    const uint64_t dV0 = sdesc_sw128(smem_u32(smem + kOffV), kKVHalf, 1024);

    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, bar, sched, k, abort_flag, idx)) return false;
        if (idx < 0) break;
        const Plan pl = make_plan<ANCH>(p, idx);
        bool pend = false;   // block j-1 awaits its PV
        bool first_pv = true;

        for (int j = 0; j <= pl.nblk; ++j) {
            const uint32_t st = g % kStages, ph = (g / kStages) & 1u;
            if (!mbar_wait_w(&bar[BAR_KV_FULL + st], ph, abort_flag, p.err)) return false;
            tc_fence_after();
            const bool now = j < pl.nblk && blk_active<ANCH>(pl, x, j);
            if (now) {
                if (j == first_blk<ANCH>(pl, x)) {
                    if (!mbar_wait_w(&bar[BAR_Q_FULL + x], q_cnt & 1u, abort_flag, p.err)) return false;
                    ++q_cnt;
                    tc_fence_after();
                }
                const uint32_t b = s_cnt & 1u;
                const uint64_t dK = dK0 + st * (kKVBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < kHD / 16; ++kk) {
                    const uint32_t offq = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    const uint32_t offk = (kk >> 2) * kKVHalf + (kk & 3) * 32;
                    umma_bf16_w(tmem + col_s(x, b), dQ + (offq >> 4), dK + (offk >> 4), kIdescS,
                                kk > 0 ? 1u : 0u);
                }
                umma_commit_w(&bar[BAR_S_FULL + 2 * x + b]);
                if (j == pl.j1[x]) umma_commit_w(&bar[BAR_Q_EMPTY + x]);
                ++s_cnt;
            }
            if (pend) {
                const uint32_t n = s_cnt - (now ? 2u : 1u);   // block j-1's S
                const uint32_t b = n & 1u;
                if (!mbar_wait_w(&bar[BAR_P_FULL + 2 * x + b], (n >> 1) & 1u, abort_flag, p.err))
                    return false;
                if (first_pv) {
                    if (!mbar_wait_w(&bar[BAR_O_FREE + x], (o_cnt & 1u) ^ 1u, abort_flag, p.err))
                        return false;
                    ++o_cnt;
                }
                tc_fence_after();
                const uint64_t dV = dV0 + st * (kKVBytes >> 4);
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk)
                    umma_bf16_ts_w(tmem + col_o(x), tmem + col_s(x, b) + kk * 8,
                                   dV + ((kk * 16 * 128) >> 4), kIdescO,
                                   (first_pv && kk == 0) ? 0u : 1u);
                first_pv = false;
                umma_commit_w(&bar[(j - 1 == pl.j1[x]) ? BAR_O_FULL + x : BAR_O_DONE + x]);
            }
            pend = now;
            umma_commit_w(&bar[BAR_KV_EMPTY + st]);
            ++g;
        }
    }
    return true;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* err) {
    return mbar_wait_w(bar, parity, abort_flag, err);
}

// ANCH: the launch has global anchors (p.S > 0); without them the anchor run
// is compiled out and the loop is the plain window / far walk.
template <bool ANCH>
__device__ bool softmax_role(const PfParams& p, uint8_t* smem, uint64_t* bar, volatile int* sched,
                             uint32_t tmem, volatile int* abort_flag, int x, int wq, int lane) {
    const int r = wq * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tO = lane_base + col_o(x);
    const float sl = p.scale_log2;
    // This warp's 4 KiB staging area for coalesced output stores.
    const uint32_t stg = smem_u32(smem + kOffStage + (x * 4 + wq) * kStageBytesPerWarp);
    uint32_t s_cnt = 0, o_cnt = 0, od_cnt = 0;

    for (int k = 0;; ++k) {
        int idx;
        if (!consume_item(p, bar, sched, k, abort_flag, idx)) return false;
        if (idx < 0) break;
        const Plan pl = make_plan<ANCH>(p, idx);
        if (!tile_active(pl, x)) continue;
        const bool far = pl.kind != kItemBand;
        int i = -1;
        if (r >= pl.rlo[x] && r < pl.nrows[x]) {
            const int rr = pl.row0 + x * kBM + r;
            i = far ? p.routed_list[(size_t)pl.b * p.N + rr] : rr;
        }
        bool write_row = i >= 0;
        if (!far && i >= 0) write_row = !(p.gate[(size_t)pl.b * p.N + i] != 0 && i >= p.W);
        const int lo = (i < 0) ? 1 : (far ? 0 : max(0, i - p.W + 1));
        const int hi = (i < 0) ? 0 : i;

        // With anchors the tile first walks its anchor run (blocks 0 .. ja1,
        // keys from 0, this row's anchors below its window being
        // [0, min(S, i-W+1))), skipping any block between the two runs.
        const int e_anc = (ANCH && i >= 0 && !far) ? min(p.S - 1, i - p.W) : -1;

        float m2 = -INFINITY, l = 0.f;
        bool first = true;
        for (int j = first_blk<ANCH>(pl, x); j <= pl.j1[x]; ++j) {
            if (ANCH && j > pl.ja1[x] && j < pl.j0[x]) continue;
            const bool anc = ANCH && j <= pl.ja1[x];
            const int key0 = blk_key0<ANCH>(pl, j);
            const int a = (anc ? 0 : lo) - key0, e = (anc ? e_anc : hi) - key0;
            const uint32_t b = s_cnt & 1u;
            if (!warp_wait(&bar[BAR_S_FULL + 2 * x + b], (s_cnt >> 1) & 1u, abort_flag, p.err))
                return false;
            tc_fence_after();
            const uint32_t tS = lane_base + col_s(x, b);
            uint32_t sr[kKB];
            tmem_ld32(tS + 0, sr);
            tmem_ld32(tS + 32, sr + 32);
            tmem_ld_wait();
            float* s = reinterpret_cast<float*>(sr);
            const bool full = a <= 0 && e >= kKB - 1;   // every key of the block visible
            // Warp-uniform classification (every lane votes, the branches
            // follow the votes, so a warp never runs two paths): a mask that
            // is one-sided for the whole warp (visible c <= e: diagonal and
            // far blocks; c >= a: window start) costs one compare and one
            // select per column; the maximum is then the same three-input
            // tree as for a full block.
            const bool all_full = __all_sync(0xffffffffu, full);
            const bool all_pre = __all_sync(0xffffffffu, a <= 0);
            const bool all_suf = __all_sync(0xffffffffu, e >= kKB - 1);
            float m8[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) m8[t] = -INFINITY;
            if (!all_full) {
                if (all_pre) {
#pragma unroll
                    for (int cc = 0; cc < kKB; ++cc) s[cc] = cc <= e ? s[cc] : -INFINITY;
                } else if (all_suf) {
#pragma unroll
                    for (int cc = 0; cc < kKB; ++cc) s[cc] = cc >= a ? s[cc] : -INFINITY;
                } else {
                    const uint32_t span = static_cast<uint32_t>(e - a);
#pragma unroll
                    for (int cc = 0; cc < kKB; ++cc) {
                        const bool ok = static_cast<uint32_t>(cc - a) <= span && e >= a;
                        s[cc] = ok ? s[cc] : -INFINITY;
                    }
                }
            }
#pragma unroll
            for (int cc = 0; cc < kKB; cc += 16)
#pragma unroll
                for (int t = 0; t < 8; ++t) m8[t] = fmax3(m8[t], s[cc + 2 * t], s[cc + 2 * t + 1]);
            const float mx = fmaxf(fmax3(m8[0], m8[1], m8[2]),
                                   fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
            // Running max in scaled log2 units; O and l are rescaled only when
            // the max grows by more than 2^8 (p stays <= 256 otherwise).
            const float mnew = fmaxf(m2, mx * sl);
            const bool resc = mnew > m2 + 8.0f;
            float alpha = 1.f;
            if (resc) {
                alpha = ex2_approx(m2 - mnew);
                m2 = mnew;
            }
            const float mb = (m2 == -INFINITY) ? 0.f : m2;
            const float2 sl2 = make_float2(sl, sl), nmb = make_float2(-mb, -mb);
            float2 r4[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) r4[t] = make_float2(0.f, 0.f);
            // p = 2^(s * scale * log2 e - m) on the MUFU (a masked key's
            // weight is exactly 0); scale-and-subtract and the row sums use
            // packed fp32 pairs.  P goes over the S columns just read.
            {
                uint32_t pk[kKB / 2];
#pragma unroll
                for (int pp = 0; pp < kKB / 2; ++pp) {
                    const float2 xv = ffma2(make_float2(s[2 * pp], s[2 * pp + 1]), sl2, nmb);
                    float2 pv;
                    pv.x = ex2_approx(xv.x);
                    pv.y = ex2_approx(xv.y);
                    r4[pp & 3] = fadd2(r4[pp & 3], pv);
                    pk[pp] = pack_bf16x2(pv.x, pv.y);
                }
                tmem_st32(tS, pk);
            }
            const float2 rs2 = fadd2(fadd2(r4[0], r4[1]), fadd2(r4[2], r4[3]));
            const float rs = rs2.x + rs2.y;
            // O may be rescaled only once the previous block's PV has landed.
            // Its commit is BAR_O_DONE phase od_cnt (every PV of the run but
            // the last commits one); that phase is waited for only when some
            // row rescales.  Skipping the wait otherwise keeps the parity test
            // unambiguous: S(j) completing implies PV(j-2) did (same issuing
            // thread, issued before it), and PV(j) needs this block's P, so
            // the barrier is at phase od_cnt or just past it.
            const bool need = resc && l > 0.f;
            const bool any_need = __any_sync(0xffffffffu, need);
            if (!first) {
                if (any_need) {
                    if (!warp_wait(&bar[BAR_O_DONE + x], od_cnt & 1u, abort_flag, p.err)) return false;
                    tc_fence_after();
                }
                ++od_cnt;
            }
            if (any_need) {
                const float f = need ? alpha : 1.f;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t orr[32];
                    tmem_ld32(tO + q4 * 32, orr);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 32; ++t) orr[t] = __float_as_uint(__uint_as_float(orr[t]) * f);
                    tmem_st32(tO + q4 * 32, orr);
                }
            }
            tmem_st_wait();
            l = l * alpha + rs;
            first = false;
            ++s_cnt;
            tc_fence_before();
            mbar_arrive(&bar[BAR_P_FULL + 2 * x + b]);
        }

        // Epilogue: O/l as bf16.  Each thread stages its row (64 columns at a
        // time) in shared memory; the warp then stores 4 whole rows per
        // instruction (8 lanes x 16 bytes per 128-byte row segment).
        if (!warp_wait(&bar[BAR_O_FULL + x], o_cnt & 1u, abort_flag, p.err)) return false;
        ++o_cnt;
        tc_fence_after();
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const unsigned long long out_row =
            (i >= 0) ? (((unsigned long long)pl.b * p.N + i) * p.Hq + pl.h) : 0ull;
        const int wflag = write_row ? 1 : 0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t orr[64];
            tmem_ld32(tO + hh * 64, orr);
            tmem_ld32(tO + hh * 64 + 32, orr + 32);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t addr = stg + lane * 128 + ((((uint32_t)u) ^ ((uint32_t)lane & 7u)) << 4);
                st_shared_v4(addr,
                             pack_bf16x2(__uint_as_float(orr[8 * u + 0]) * inv, __uint_as_float(orr[8 * u + 1]) * inv),
                             pack_bf16x2(__uint_as_float(orr[8 * u + 2]) * inv, __uint_as_float(orr[8 * u + 3]) * inv),
                             pack_bf16x2(__uint_as_float(orr[8 * u + 4]) * inv, __uint_as_float(orr[8 * u + 5]) * inv),
                             pack_bf16x2(__uint_as_float(orr[8 * u + 6]) * inv, __uint_as_float(orr[8 * u + 7]) * inv));
            }
            __syncwarp();
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int row = it * 4 + (lane >> 3);
                const uint32_t u = lane & 7;
                const unsigned long long orow = __shfl_sync(0xffffffffu, out_row, row);
                const int wf = __shfl_sync(0xffffffffu, wflag, row);
                const uint4 val = ld_shared_v4(stg + row * 128 + ((u ^ ((uint32_t)row & 7u)) << 4));
                if (wf) *reinterpret_cast<uint4*>(p.o + orow * kHD + hh * 64 + u * 8) = val;
            }
            __syncwarp();
        }
        if (write_row && p.lse) p.lse[out_row] = (m2 + __log2f(l)) * 0.69314718055994531f;
        tc_fence_before();
        mbar_arrive(&bar[BAR_O_FREE + x]);
    }
    return true;
}

template <bool ANCH>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PfParams p) {
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
            mbar_init(&bar[BAR_O_DONE + x], 1);
            mbar_init(&bar[BAR_O_FULL + x], 1);
            mbar_init(&bar[BAR_O_FREE + x], kBM);
        }
        for (int sb = 0; sb < 4; ++sb) {
            mbar_init(&bar[BAR_S_FULL + sb], 1);
            mbar_init(&bar[BAR_P_FULL + sb], kBM);
        }
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&bar[BAR_KV_FULL + st], 1);
            mbar_init(&bar[BAR_KV_EMPTY + st], 2);   // one commit per MMA warp
        }
        for (int st = 0; st < kSched; ++st) {
            mbar_init(&bar[BAR_SCHED_FULL + st], 1);
            mbar_init(&bar[BAR_SCHED_EMPTY + st], kSchedConsumers);
        }
        mbar_init(&bar[BAR_DRAIN], 2);
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
    // Launched as a programmatic dependent of the schedule: everything above
    // overlaps it; its work list, far-row list and tile prefixes are read
    // only after this wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp < 8) {
        warpgroup_reg_inc<kRegsSoftmax>();
        softmax_role<ANCH>(p, smem, bar, sched, tmem, abort_flag, warp >> 2, warp & 3, lane);
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
        bool q_tma_last[2] = {false, false};
        if (!producer<ANCH>(p, smem, bar, sched, abort_flag, g, q_issued, q_tma_last)) {
            drain_loads(&bar[BAR_KV_FULL], g);
            for (int x = 0; x < 2; ++x)
                if (q_tma_last[x]) mbar_drain(&bar[BAR_Q_FULL + x], (q_issued[x] - 1) & 1u);
        }
        __syncwarp();
    } else if (warp == 9 || warp == 11) {
        mma_issuer<ANCH>(p, smem, bar, sched, tmem, abort_flag, warp == 9 ? 0 : 1);
        // Every MMA both warps issued has completed once this phase completes.
        umma_commit_w(&bar[BAR_DRAIN]);
        mbar_drain(&bar[BAR_DRAIN], 0);
        __syncwarp();
    } else if (warp == 10) {
        q_gatherer<ANCH>(p, smem, bar, sched, abort_flag, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_prefill_tc(const TcAttnArgs& a, const int* tile_prefix, unsigned int* err,
                              int num_sms, cudaStream_t s) {
    PfParams p;
    memset(&p, 0, sizeof(p));
    const uint64_t N = a.N, B = a.B;
    bool ok = make_tmap_4d_bf16(&p.tm_q, a.q, kHD, a.Hq, N, B, 64, kBM) &&
              make_tmap_4d_bf16(&p.tm_k, a.k, kHD, a.Hkv, N, B, 64, kKB) &&
              make_tmap_4d_bf16(&p.tm_v, a.v, kHD, a.Hkv, N, B, 64, kKB);
    if (!ok) return cudaErrorInvalidValue;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.routed_list = a.routed_list;
    p.routed_count = a.routed_count;
    p.tile_prefix = tile_prefix;
    p.n_items = a.n_items;
    p.next_item = const_cast<int*>(a.n_items) + 1;
    p.items = a.items;
    p.gate = a.gate;
    p.o = static_cast<__nv_bfloat16*>(a.o);
    p.lse = a.lse;
    p.err = err;
    p.B = a.B;
    p.N = a.N;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.W = a.W;
    p.S = a.n_anchor;
    p.NT = (a.N + kBM - 1) / kBM;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    static std::atomic<uint64_t> smem_plain{0}, smem_anchored{0};
    cudaError_t e = p.S > 0 ? allow_dynamic_smem(prefill_kernel<true>, kSmemBytes, smem_anchored)
                            : allow_dynamic_smem(prefill_kernel<false>, kSmemBytes, smem_plain);
    if (e != cudaSuccess) return e;
    // A programmatic dependent launch of the schedule kernel before it on the
    // stream: the CTAs start (TMEM, barriers) while the schedule runs and wait
    // for its grid before reading the work list.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = p.S > 0 ? cudaLaunchKernelEx(&cfg, prefill_kernel<true>, p)
                : cudaLaunchKernelEx(&cfg, prefill_kernel<false>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t prefill_set_wait_limit(uint64_t ns) { return set_wait_limit_of_unit(ns); }

}  // namespace swi
