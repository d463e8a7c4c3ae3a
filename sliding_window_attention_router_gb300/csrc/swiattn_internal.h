// Internal declarations shared by the translation units of libswiattn.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>
#include <cstdint>

namespace swi {

// Device error word bits (OR-ed by kernels, read by swiattn_get_device_error).
constexpr unsigned int kDevErrTimeout = 1u;
constexpr unsigned int kDevErrLayout = 2u;   // shared memory not laid out as a kernel requires
constexpr unsigned int kDevErrInput = 4u;    // a device-resident input was out of range

// A healthy wait in these kernels lasts microseconds; after this long a
// kernel gives up, flags a timeout and returns (the default; a test may lower
// it through swiattn_set_wait_limit_ns).  Waits while aborting keep their own
// fixed limit.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainLimitNs = 100000000ull;   // 0.1 s, waits while aborting

// Per translation unit setters of the wait limit (current device; 0 restores
// the default): the routed prefill, the dual-branch forward, the backward.
cudaError_t prefill_set_wait_limit(uint64_t ns);
cudaError_t dual_set_wait_limit(uint64_t ns);
cudaError_t bwd_set_wait_limit(uint64_t ns);

// Lets `kernel` use `bytes` of dynamic shared memory on the current device.
// The attribute belongs to the device's context, so it is set once per
// device (devices 0-63 are remembered in `done`; others set it every call),
// and concurrent callers may both set it, which is harmless.
template <typename K>
cudaError_t allow_dynamic_smem(K kernel, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// ------------------------------------------------------------ tiling --------
constexpr int kBM = 128;   // query rows per tile (TMEM lanes)
constexpr int kBN = 128;   // keys per tile
constexpr int kHD = 128;   // head dim of the tensor-core path

// Work item kinds of the routed-prefill schedule.
constexpr int kItemBand = 0;   // 256 consecutive rows, window keys, writes non-far rows
constexpr int kItemFar = 1;    // 256 compacted routed rows, causal keys [0, i]
constexpr int kItemFarA = 2;   // the same pair's first 128 far rows alone
constexpr int kItemFarB = 3;   // the same pair's last 128 far rows alone

struct WorkItem {
    int kind, b, h, tile;
};

// Far rows fill 128-row tiles in ascending row order; the first tile holds
// the remainder of the count R, its first far_front(R) slots empty, so the
// part-filled tile holds the earliest rows (the shortest key prefix).
__host__ __device__ inline int far_front(int R) { return (kBM - R % kBM) % kBM; }

// Workspace layout of swiattn_prefill (byte offsets from a 256-aligned base).
struct PrefillWs {
    size_t routed_list;   // int32 [B*N]   far rows of each batch, ascending
    size_t routed_count;  // int32 [B]
    size_t tile_prefix;   // int32 [B*(NT+1)] far rows before each 128-row tile
    size_t far_last;      // int32 [B*NT]     last row of each far tile (-1 past the last)
    size_t n_items;       // int32 [4]
    size_t items;         // WorkItem [max_items]
    size_t total;
    int max_items;
};
PrefillWs prefill_ws_layout(int B, int N, int Hq, int d);

struct DecodeWs {
    size_t part;   // float [B * max_chunks * Hq * (d+2)]
    size_t claim;  // int: chunk counter of the split kernel's persistent CTAs (cleared per call)
    size_t total;
    int max_chunks;
    int chunk;
};
// S: global anchors (extra anchor chunks per sequence; 0 for plain decode).
DecodeWs decode_ws_layout(int B, int Lmax, int Hq, int d, int S);

struct DualWs {
    size_t lse_full;  // float [B*N*Hq] (fp32 path: lse of both branches)
    size_t lse_swa;   // float [B*N*Hq]
    size_t mse_part;  // float [B*N*Hq]
    size_t snap;      // float [B*N*Hq*128] O_SWA rows, fp32 (tensor-core path)
    size_t counter;   // int32 work counter
    size_t total;
};
DualWs dual_ws_layout(int B, int N, int Hq, int d, int dtype);

// ------------------------------------------------------------ launchers -----
// Each returns cudaSuccess or the launch error.
cudaError_t launch_route(const void* h, const void* w, float bias, int64_t tokens, int d_model,
                         int dtype, float* logits, uint8_t* gate, cudaStream_t s);

// Far-row lists, tile prefix counts and the cost-sorted work list of the
// routed prefill, in one single-CTA launch.  S: global anchors of window rows
// (adds their key blocks to band items' cost).  grid: CTAs of the attention
// launch (a far pair costing more than 1.25 x a CTA's mean share is listed as
// two one-tile items).
cudaError_t launch_schedule(const uint8_t* gate, int B, int N, int Hq, int W, int S, int grid,
                            const PrefillWs& L, char* ws, cudaStream_t s);

// Router GEMV over the B*N tokens (logits, gates) fused with the schedule
// above: the last CTA to finish plans over the gates.  ticket: a 4-byte
// counter in device memory, zeroed here before the launch.
cudaError_t launch_route_plan(const void* h, const void* w, float bias, int d_model, int dtype,
                              float* logits, uint8_t* gate, int B, int N, int Hq, int W, int S,
                              const PrefillWs& L, char* ws, unsigned int* ticket, int num_sms,
                              cudaStream_t s);

struct TcAttnArgs {
    const void* q;     // [B,N,Hq,128] bf16
    const void* k;     // [B,N,Hkv,128]
    const void* v;
    const int* routed_list;
    const int* routed_count;
    const int* n_items;
    const WorkItem* items;
    const uint8_t* gate;
    const float* logits;   // dual: for o_gated
    void* o;               // prefill output / dual o_full
    void* o_swa;           // dual
    void* o_gated;         // dual, nullable
    float* lse;            // prefill, or dual's lse of the gated output; nullable
    float* mse_part;       // dual
    float* snap;           // dual: fp32 O_SWA rows
    int* counter;          // dual: work counter (zeroed by the launcher)
    int B, N, Hq, Hkv, W;
    int n_anchor;          // prefill: global anchors of window rows (0: none)
    float scale;
};

// Dual-branch forward, two query tiles per CTA (the launcher records the
// profile events around the kernel itself).
cudaError_t launch_dual_tc(const TcAttnArgs& a, unsigned int* err, int num_sms, cudaStream_t s);

// Routed prefill, two query tiles per CTA (work items from launch_schedule).
cudaError_t launch_prefill_tc(const TcAttnArgs& a, const int* tile_prefix, unsigned int* err,
                              int num_sms, cudaStream_t s);

// S: global anchors of window rows (0: none).
cudaError_t launch_simt_attention(const void* q, const void* k, const void* v,
                                  const uint8_t* gate, int force, void* o, float* lse, int B,
                                  int N, int Hq, int Hkv, int d, int W, int S, float scale,
                                  int dtype, cudaStream_t s);

cudaError_t launch_dual_epilogue_f32(const float* o_full, const float* o_swa,
                                     const float* logits, const float* nll, float* o_gated,
                                     const float* lse_full, const float* lse_swa, float* lse_gated,
                                     float* mse, float* gamma, float* reg, int B, int N, int Hq,
                                     int d, float gamma_base, float eps, float alpha,
                                     cudaStream_t s);

cudaError_t launch_dual_epilogue_parts(const float* mse_part, const float* logits,
                                       const float* nll, float* mse, float* gamma, float* reg,
                                       int B, int N, int Hq, float gamma_base, float eps,
                                       float alpha, cudaStream_t s);

// SWIATTN_OK when the decode split kernel for these sizes fits one block on
// the current device (one thread per 16 bytes of a token row, all KV heads;
// the kernel's register use caps the block below 1024 threads for most
// kinds), SWIATTN_EUNSUPPORTED when it does not.  When the kernel's
// attributes cannot be read it answers SWIATTN_OK and the launch decides.
// Hq/Hkv must be 1, 2, 4 or 8.
int decode_block_check(int dtype, int d, int Hq, int Hkv, bool paged);

// err: device error word (a length outside [1, Lmax] is clamped and reported).
cudaError_t launch_decode(const void* q, const void* kc, const void* vc, const int32_t* seq_lens,
                          const uint8_t* gate, void* o, float* lse, int B, int Lmax, int Hq,
                          int Hkv, int d, int W, int S, float scale, int dtype,
                          const DecodeWs& L, char* ws, unsigned int* err, cudaStream_t s);

// ------------------------------------------------------------ backward ------
// Far-row scan alone (one CTA per batch): routed_list/routed_count/
// tile_prefix as in PrefillWs.
cudaError_t launch_far_scan(const uint8_t* gate, int B, int N, int W, int* routed_list,
                            int* routed_count, int* tile_prefix, cudaStream_t s);

// Work item of the tensor-core backward kernels (32 bytes).
//  kBwdKV:    one 128-key block t of (b, kv head h); for each query head of the
//             group it visits the band query tiles starting at 128*t + 128*u,
//             u < a0, then the far (compacted) tiles [a1, a2).
//  kBwdQBand: query tile t (rows 128*t ...) of (b, query head h), window keys.
//  kBwdQFar:  compacted far tile t of (b, h), keys [0, max i].
constexpr int kBwdKV = 0;
constexpr int kBwdQBand = 1;
constexpr int kBwdQFar = 2;
struct BwdItem {
    int kind, b, h, t;
    int a0, a1, a2, cost;
};
static_assert(sizeof(BwdItem) == 32, "BwdItem is read as two int4");

// Rows of a compacted far tile past the routed count carry this row index.
constexpr int kNoRow = -(1 << 30);

// Workspace layout of swiattn_prefill_backward (tensor-core path; byte
// offsets from a 256-aligned base).  Npad = N rounded up to 128.
struct BwdWs {
    size_t routed_list;   // int32 [B*N]
    size_t routed_count;  // int32 [B]
    size_t tile_prefix;   // int32 [B*(NT+1)]
    size_t rowidx;        // int32 [B*Npad]  far rows (compacted), kNoRow padded per tile
    size_t d_band;        // f32 [B*Hq*Npad] D_i = <dO_i, O_i>, head-major
    size_t l_band;        // f32 [B*Hq*Npad] lse_i * log2(e)
    size_t d_far;         // f32 [B*Hq*Npad] the same for compacted far rows
    size_t l_far;         // f32 [B*Hq*Npad]
    size_t qc;            // bf16 [B*Npad*Hq*128] compacted q of far rows (zero pads)
    size_t doc;           // bf16 [B*Npad*Hq*128] compacted dO of far rows
    size_t counters;      // int32 [4]: n_kv, next_kv, n_q, next_q
    size_t items_kv;      // BwdItem [max_kv]
    size_t items_q;       // BwdItem [max_q]
    size_t total;
    int Npad, max_kv, max_q;
};
BwdWs bwd_ws_layout(int B, int N, int Hq, int Hkv);

// Scan, row statistics, compaction and work lists of the backward.
cudaError_t launch_bwd_schedule(const uint8_t* gate, const void* q, const void* o,
                                const float* lse, const void* d_o, int B, int N, int Hq,
                                int Hkv, int W, const BwdWs& L, char* ws, int num_sms,
                                cudaStream_t s);

struct TcBwdArgs {
    const void* q;     // [B,N,Hq,128] bf16
    const void* k;     // [B,N,Hkv,128]
    const void* v;
    const void* d_o;   // [B,N,Hq,128]
    const uint8_t* gate;
    void* dq;          // [B,N,Hq,128] bf16
    void* dk;          // [B,N,Hkv,128]
    void* dv;
    const BwdWs* L;
    char* ws;
    int B, N, Hq, Hkv, W;
    float scale;
};
cudaError_t launch_bwd_dkdv(const TcBwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s);
cudaError_t launch_bwd_dq(const TcBwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s);

// fp32 backward on CUDA cores (dtype SWIATTN_F32, d in {64, 128}); ws holds
// B*N*Hq floats.
cudaError_t launch_simt_backward(const float* q, const float* k, const float* v,
                                 const uint8_t* gate, const float* o, const float* lse,
                                 const float* d_o, float* dq, float* dk, float* dv, int B, int N,
                                 int Hq, int Hkv, int d, int W, float scale, float* ws,
                                 cudaStream_t s);

// Router backward (straight-through gate + regulariser, then the linear map).
int64_t route_bwd_chunks(int64_t tokens);
cudaError_t launch_route_backward(const void* h, const void* w, const float* logits,
                                  const void* o_full, const void* o_swa, const void* d_o,
                                  const float* gamma, const float* d_reg, int64_t tokens, int hd,
                                  int d_model, int dtype, float* d_logits, void* dh, float* dw,
                                  float* db, float* ws, cudaStream_t s);

// Decode over a paged cache: k/v pages [num_pages, 1 << page_lg, Hkv, d],
// block_table [B, max_pages]; bad table entries are flagged in *err.
cudaError_t launch_decode_paged(const void* q, const void* kp, const void* vp,
                                const int32_t* block_table, const int32_t* seq_lens,
                                const uint8_t* gate, void* o, float* lse, int B, int max_pages,
                                int page_lg, int num_pages, int Hq, int Hkv, int d, int W, int S,
                                float scale, int dtype, const DecodeWs& L, char* ws,
                                unsigned int* err, cudaStream_t s);

// Timing hook around the dominant kernel of a call (no-ops unless set).
void prof_start(cudaStream_t s);
void prof_stop(cudaStream_t s);

// TMA descriptor creation through the driver entry point (no libcuda link).
bool make_tmap_4d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t d3, uint32_t box0, uint32_t box2);

}  // namespace swi
