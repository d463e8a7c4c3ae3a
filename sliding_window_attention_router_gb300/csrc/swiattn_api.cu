// C ABI of libswiattn: argument validation, workspace carving and launches.
// Declarations and the contract of every entry point are in include/swiattn.h.

#include "swiattn.h"
#include "swiattn_internal.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstring>
#include <mutex>

namespace swi {
namespace {

// Device error word: kernels OR kDevErrTimeout into it when a bounded wait
// expires, kDevErrLayout when their shared memory is not laid out as needed.  Host code reaches it through cudaGetSymbolAddress, once per device.
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];

struct DeviceInfo {
    unsigned int* err;
    int sms;
};

bool device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return false;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return false;
        g_err_ptr[dev] = static_cast<unsigned int*>(p);
        g_num_sms[dev] = sms;
    }
    out.err = g_err_ptr[dev];
    out.sms = g_num_sms[dev];
    return true;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Profiling hook events: set by one thread, read by every launching thread.
std::atomic<cudaEvent_t> g_prof_start{nullptr}, g_prof_stop{nullptr};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

int launched(cudaError_t e) { return e == cudaSuccess ? SWIATTN_OK : SWIATTN_ECUDA; }

bool attn_shape_ok(int B, int N, int Hq, int Hkv, int d, int W) {
    return B > 0 && N > 0 && Hq > 0 && Hkv > 0 && W > 0 && Hq % Hkv == 0 && (d == 64 || d == 128) &&
           (int64_t)B * N * Hq * d < (int64_t(1) << 40);
}

}  // namespace

void prof_start(cudaStream_t s) {
    cudaEvent_t a = g_prof_start.load(std::memory_order_acquire);
    if (a && g_prof_stop.load(std::memory_order_acquire)) cudaEventRecord(a, s);
}
void prof_stop(cudaStream_t s) {
    cudaEvent_t b = g_prof_stop.load(std::memory_order_acquire);
    if (b && g_prof_start.load(std::memory_order_acquire)) cudaEventRecord(b, s);
}

bool make_tmap_4d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t d3, uint32_t box0, uint32_t box2) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {d0, d1, d2, d3};
    const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
    const cuuint32_t box[4] = {box0, 1, box2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

DualWs dual_ws_layout(int B, int N, int Hq, int d, int dtype) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    DualWs L;
    L.lse_full = L.lse_swa = L.mse_part = L.snap = L.counter = L.total = 0;
    const size_t rows = (size_t)B * N * Hq;
    if (dtype != SWIATTN_BF16) {
        L.lse_swa = up(sizeof(float) * rows);
        L.total = up(L.lse_swa + sizeof(float) * rows);
        return L;
    }
    L.snap = up(sizeof(float) * rows);
    L.counter = up(L.snap + sizeof(float) * rows * (size_t)d);
    L.total = up(L.counter + sizeof(int));
    return L;
}

}  // namespace swi

using namespace swi;

extern "C" {

const char* swiattn_status_string(int status) {
    switch (status) {
        case SWIATTN_OK: return "SWIATTN_OK";
        case SWIATTN_EINVAL: return "SWIATTN_EINVAL";
        case SWIATTN_EUNSUPPORTED: return "SWIATTN_EUNSUPPORTED";
        case SWIATTN_ECUDA: return "SWIATTN_ECUDA";
        case SWIATTN_ETIMEOUT: return "SWIATTN_ETIMEOUT";
        default: return "SWIATTN_UNKNOWN";
    }
}

void swiattn_set_profile_events(void* start, void* stop) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_prof_start.store(static_cast<cudaEvent_t>(start), std::memory_order_release);
    g_prof_stop.store(static_cast<cudaEvent_t>(stop), std::memory_order_release);
}

int swiattn_set_wait_limit_ns(uint64_t ns) {
    if (prefill_set_wait_limit(ns) != cudaSuccess || dual_set_wait_limit(ns) != cudaSuccess ||
        bwd_set_wait_limit(ns) != cudaSuccess)
        return SWIATTN_ECUDA;
    return SWIATTN_OK;
}

int swiattn_num_sms(void) {
    DeviceInfo di;
    return device_info(di) ? di.sms : -1;
}

int swiattn_get_device_error(void* stream) {
    DeviceInfo di;
    if (!device_info(di)) return SWIATTN_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int host = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SWIATTN_ECUDA;
    if (cudaMemcpy(&host, di.err, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SWIATTN_ECUDA;
    if (host) {
        const unsigned int zero = 0;
        if (cudaMemcpy(di.err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return SWIATTN_ECUDA;
    }
    if (host & kDevErrTimeout) return SWIATTN_ETIMEOUT;
    if (host & kDevErrInput) return SWIATTN_EINVAL;
    return host ? SWIATTN_ECUDA : SWIATTN_OK;
}

int swiattn_route(const void* h, const void* w, float bias, int64_t tokens, int d_model, int dtype,
                  float* logits, uint8_t* gate, void* stream) {
    if (tokens < 0 || d_model <= 0) return SWIATTN_EINVAL;
    if (dtype != SWIATTN_BF16 && dtype != SWIATTN_F32) return SWIATTN_EINVAL;
    if (d_model % (dtype == SWIATTN_BF16 ? 8 : 4) != 0) return SWIATTN_EINVAL;
    if (tokens == 0) return SWIATTN_OK;
    if (!h || !w || !logits || !gate || !aligned16(h) || !aligned16(w)) return SWIATTN_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    prof_start(s);
    const cudaError_t e = launch_route(h, w, bias, tokens, d_model, dtype, logits, gate, s);
    prof_stop(s);
    return launched(e);
}

size_t swiattn_prefill_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype) {
    if (!attn_shape_ok(B, N, Hq, Hkv, d, W)) return 0;
    if (dtype != SWIATTN_BF16) return 256;   // the fp32 path needs none
    return prefill_ws_layout(B, N, Hq, d).total;
}

int swiattn_prefill(const void* q, const void* k, const void* v, const uint8_t* gate, void* o,
                    float* lse, int B, int N, int Hq, int Hkv, int d, int W, float scale,
                    int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    return swiattn_prefill_anchored(q, k, v, gate, o, lse, B, N, Hq, Hkv, d, W, 0, scale, dtype,
                                    workspace, workspace_bytes, stream);
}

namespace {

int prefill_args_ok(const void* q, const void* k, const void* v, const void* o, int B, int N,
                    int Hq, int Hkv, int d, int W, int n_anchor, float scale) {
    if (!attn_shape_ok(B, N, Hq, Hkv, d, W) || n_anchor < 0) return SWIATTN_EINVAL;
    if (!q || !k || !v || !o) return SWIATTN_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SWIATTN_EINVAL;
    if (!(scale > 0.f)) return SWIATTN_EINVAL;
    return SWIATTN_OK;
}

// The attention launch of the tensor-core prefill, once the schedule has been
// enqueued on s (workspace laid out by prefill_ws_layout).
int launch_prefill_after_plan(const void* q, const void* k, const void* v, const uint8_t* gate,
                              void* o, float* lse, int B, int N, int Hq, int Hkv, int W,
                              int n_anchor, float scale, const PrefillWs& L, char* ws,
                              const DeviceInfo& di, cudaStream_t s) {
    TcAttnArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k;
    a.v = v;
    a.routed_list = reinterpret_cast<const int*>(ws + L.routed_list);
    a.routed_count = reinterpret_cast<const int*>(ws + L.routed_count);
    a.n_items = reinterpret_cast<const int*>(ws + L.n_items);
    a.items = reinterpret_cast<const WorkItem*>(ws + L.items);
    a.gate = gate;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.N = N;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.W = W;
    a.n_anchor = n_anchor;
    a.scale = scale;
    prof_start(s);
    cudaError_t e = launch_prefill_tc(a, reinterpret_cast<const int*>(ws + L.tile_prefix), di.err,
                                      di.sms, s);
    prof_stop(s);
    return launched(e);
}

}  // namespace

int swiattn_prefill_anchored(const void* q, const void* k, const void* v, const uint8_t* gate,
                             void* o, float* lse, int B, int N, int Hq, int Hkv, int d, int W,
                             int n_anchor, float scale, int dtype, void* workspace,
                             size_t workspace_bytes, void* stream) {
    const int ok = prefill_args_ok(q, k, v, o, B, N, Hq, Hkv, d, W, n_anchor, scale);
    if (ok != SWIATTN_OK) return ok;
    if (!gate) return SWIATTN_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SWIATTN_F32) {
        return launched(launch_simt_attention(q, k, v, gate, -1, o, lse, B, N, Hq, Hkv, d, W,
                                              n_anchor, scale, dtype, s));
    }
    if (dtype != SWIATTN_BF16) return SWIATTN_EINVAL;
    if (d != kHD) return SWIATTN_EUNSUPPORTED;
    const PrefillWs L = prefill_ws_layout(B, N, Hq, d);
    if (!workspace || !aligned256(workspace) || workspace_bytes < L.total) return SWIATTN_EINVAL;
    DeviceInfo di;
    if (!device_info(di)) return SWIATTN_ECUDA;
    char* ws = static_cast<char*>(workspace);
    if (launch_schedule(gate, B, N, Hq, W, n_anchor, di.sms, L, ws, s) != cudaSuccess)
        return SWIATTN_ECUDA;
    return launch_prefill_after_plan(q, k, v, gate, o, lse, B, N, Hq, Hkv, W, n_anchor, scale, L,
                                     ws, di, s);
}

namespace {

// Device staging of swiattn_prefill_host, after the prefill workspace.
struct HostStage {
    size_t q, k, v, gate, o, lse, total;
};
HostStage host_stage_layout(size_t base, int B, int N, int Hq, int Hkv, int d, int esize) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t rows = (size_t)B * N;
    HostStage H;
    H.q = up(base);
    H.k = up(H.q + rows * Hq * d * esize);
    H.v = up(H.k + rows * Hkv * d * esize);
    H.gate = up(H.v + rows * Hkv * d * esize);
    H.o = up(H.gate + rows);
    H.lse = up(H.o + rows * Hq * d * esize);
    H.total = up(H.lse + rows * Hq * sizeof(float));
    return H;
}

}  // namespace

size_t swiattn_prefill_host_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype) {
    const size_t base = swiattn_prefill_workspace(B, N, Hq, Hkv, d, W, dtype);
    if (base == 0 || (dtype != SWIATTN_BF16 && dtype != SWIATTN_F32)) return 0;
    return host_stage_layout(base, B, N, Hq, Hkv, d, dtype == SWIATTN_BF16 ? 2 : 4).total;
}

int swiattn_prefill_host(const void* q_host, const void* k_host, const void* v_host,
                         const uint8_t* gate_host, void* o_host, float* lse_host, int B, int N,
                         int Hq, int Hkv, int d, int W, int n_anchor, float scale, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream) {
    if (dtype != SWIATTN_BF16 && dtype != SWIATTN_F32) return SWIATTN_EINVAL;
    const size_t need = swiattn_prefill_host_workspace(B, N, Hq, Hkv, d, W, dtype);
    if (need == 0 || n_anchor < 0 || !(scale > 0.f)) return SWIATTN_EINVAL;
    if (!q_host || !k_host || !v_host || !gate_host || !o_host) return SWIATTN_EINVAL;
    if (!workspace || !aligned256(workspace) || workspace_bytes < need) return SWIATTN_EINVAL;
    const int es = dtype == SWIATTN_BF16 ? 2 : 4;
    const size_t base = swiattn_prefill_workspace(B, N, Hq, Hkv, d, W, dtype);
    const HostStage H = host_stage_layout(base, B, N, Hq, Hkv, d, es);
    char* ws = static_cast<char*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t rows = (size_t)B * N;
    const size_t qb = rows * Hq * d * es, kvb = rows * Hkv * d * es;
    if (cudaMemcpyAsync(ws + H.gate, gate_host, rows, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(ws + H.q, q_host, qb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(ws + H.k, k_host, kvb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(ws + H.v, v_host, kvb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return SWIATTN_ECUDA;
    float* lse_dev = lse_host ? reinterpret_cast<float*>(ws + H.lse) : nullptr;
    const int rc = swiattn_prefill_anchored(ws + H.q, ws + H.k, ws + H.v,
                                            reinterpret_cast<const uint8_t*>(ws + H.gate),
                                            ws + H.o, lse_dev, B, N, Hq, Hkv, d, W, n_anchor, scale,
                                            dtype, ws, base, stream);
    if (rc != SWIATTN_OK) return rc;
    if (cudaMemcpyAsync(o_host, ws + H.o, qb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SWIATTN_ECUDA;
    if (lse_host && cudaMemcpyAsync(lse_host, lse_dev, rows * Hq * sizeof(float),
                                    cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SWIATTN_ECUDA;
    return SWIATTN_OK;
}

size_t swiattn_route_prefill_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype) {
    const size_t base = swiattn_prefill_workspace(B, N, Hq, Hkv, d, W, dtype);
    if (base == 0 || dtype != SWIATTN_BF16) return base;
    return base + 256;   // the ticket of the fused router + schedule kernel
}

int swiattn_route_prefill(const void* h, const void* w, float bias, int d_model, const void* q,
                          const void* k, const void* v, void* o, float* lse, float* logits,
                          uint8_t* gate, int B, int N, int Hq, int Hkv, int d, int W, int n_anchor,
                          float scale, int dtype, void* workspace, size_t workspace_bytes,
                          void* stream) {
    const int ok = prefill_args_ok(q, k, v, o, B, N, Hq, Hkv, d, W, n_anchor, scale);
    if (ok != SWIATTN_OK) return ok;
    if (dtype != SWIATTN_BF16 && dtype != SWIATTN_F32) return SWIATTN_EINVAL;
    if (d_model <= 0 || d_model % (dtype == SWIATTN_BF16 ? 8 : 4) != 0) return SWIATTN_EINVAL;
    if (!h || !w || !logits || !gate || !aligned16(h) || !aligned16(w)) return SWIATTN_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t tokens = (int64_t)B * N;
    if (dtype == SWIATTN_F32) {
        if (launch_route(h, w, bias, tokens, d_model, dtype, logits, gate, s) != cudaSuccess)
            return SWIATTN_ECUDA;
        return launched(launch_simt_attention(q, k, v, gate, -1, o, lse, B, N, Hq, Hkv, d, W,
                                              n_anchor, scale, dtype, s));
    }
    if (d != kHD) return SWIATTN_EUNSUPPORTED;
    const PrefillWs L = prefill_ws_layout(B, N, Hq, d);
    if (!workspace || !aligned256(workspace) || workspace_bytes < L.total + 256)
        return SWIATTN_EINVAL;
    DeviceInfo di;
    if (!device_info(di)) return SWIATTN_ECUDA;
    char* ws = static_cast<char*>(workspace);
    unsigned int* ticket = reinterpret_cast<unsigned int*>(ws + L.total);
    if (launch_route_plan(h, w, bias, d_model, dtype, logits, gate, B, N, Hq, W, n_anchor, L, ws,
                          ticket, di.sms, s) != cudaSuccess)
        return SWIATTN_ECUDA;
    return launch_prefill_after_plan(q, k, v, gate, o, lse, B, N, Hq, Hkv, W, n_anchor, scale, L,
                                     ws, di, s);
}

size_t swiattn_decode_workspace(int B, int Lmax, int Hq, int Hkv, int d, int W, int dtype) {
    return swiattn_decode_anchored_workspace(B, Lmax, Hq, Hkv, d, W, 0, dtype);
}

size_t swiattn_decode_anchored_workspace(int B, int Lmax, int Hq, int Hkv, int d, int W,
                                         int n_anchor, int dtype) {
    (void)dtype;
    if (!attn_shape_ok(B, Lmax, Hq, Hkv, d, W) || n_anchor < 0) return 0;
    return decode_ws_layout(B, Lmax, Hq, d, n_anchor).total;
}

namespace {

int decode_args_ok(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                   const uint8_t* gate, const void* o, int B, int Lmax, int Hq, int Hkv, int d,
                   int W, int S, float scale, int dtype) {
    if (!attn_shape_ok(B, Lmax, Hq, Hkv, d, W) || S < 0) return SWIATTN_EINVAL;
    if (dtype != SWIATTN_BF16 && dtype != SWIATTN_F32) return SWIATTN_EINVAL;
    if (!q || !k || !v || !seq_lens || !gate || !o) return SWIATTN_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return SWIATTN_EINVAL;
    if (!(scale > 0.f)) return SWIATTN_EINVAL;
    const int G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SWIATTN_EUNSUPPORTED;
    if ((int64_t)Hkv * d / (dtype == SWIATTN_BF16 ? 8 : 4) > 1024) return SWIATTN_EUNSUPPORTED;
    if (B > 65535) return SWIATTN_EUNSUPPORTED;
    if (Lmax > (1 << 30)) return SWIATTN_EUNSUPPORTED;
    return SWIATTN_OK;
}

// Scratch of swiattn_decode_noalloc: its split-KV partials live in this fixed
// device array instead of a caller workspace.  Every GPU that loads the
// library holds it (16 MiB) until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices];

// Device address of g_decode_scratch on the current device.  In host code the
// array's name only stands in for it, so the address is looked up once per
// device, with that device current.
float* decode_scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = static_cast<float*>(ptr);
    }
    return g_scratch_ptr[dev];
}

}  // namespace

int swiattn_decode_anchored(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* seq_lens, const uint8_t* gate, void* o, float* lse,
                            int B, int Lmax, int Hq, int Hkv, int d, int W, int n_anchor,
                            float scale, int dtype, void* workspace, size_t workspace_bytes,
                            void* stream) {
    const int st = decode_args_ok(q, k_cache, v_cache, seq_lens, gate, o, B, Lmax, Hq, Hkv, d, W,
                                  n_anchor, scale, dtype);
    if (st != SWIATTN_OK) return st;
    const DecodeWs L = decode_ws_layout(B, Lmax, Hq, d, n_anchor);
    if (!workspace || !aligned256(workspace) || workspace_bytes < L.total) return SWIATTN_EINVAL;
    DeviceInfo di;
    if (!device_info(di)) return SWIATTN_ECUDA;
    const int fit = decode_block_check(dtype, d, Hq, Hkv, false);
    if (fit != SWIATTN_OK) return fit;
    return launched(launch_decode(q, k_cache, v_cache, seq_lens, gate, o, lse, B, Lmax, Hq, Hkv,
                                  d, W, n_anchor, scale, dtype, L, static_cast<char*>(workspace),
                                  di.err, static_cast<cudaStream_t>(stream)));
}

int swiattn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
                   const uint8_t* gate, void* o, float* lse, int B, int Lmax, int Hq, int Hkv,
                   int d, int W, float scale, int dtype, void* workspace, size_t workspace_bytes,
                   void* stream) {
    return swiattn_decode_anchored(q, k_cache, v_cache, seq_lens, gate, o, lse, B, Lmax, Hq, Hkv,
                                   d, W, 0, scale, dtype, workspace, workspace_bytes, stream);
}

int swiattn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, const uint8_t* gate, void* o, float* lse,
                           int B, int Lmax, int Hq, int Hkv, int d, int W, float scale, int dtype,
                           void* stream) {
    const int st = decode_args_ok(q, k_cache, v_cache, seq_lens, gate, o, B, Lmax, Hq, Hkv, d, W,
                                  0, scale, dtype);
    if (st != SWIATTN_OK) return st;
    const DecodeWs L = decode_ws_layout(B, Lmax, Hq, d, 0);
    // The partials of this call must fit the fixed scratch array.
    if (L.total > kNoAllocScratchBytes) return SWIATTN_EINVAL;
    DeviceInfo di;
    if (!device_info(di)) return SWIATTN_ECUDA;
    float* scratch = decode_scratch_on_current_device();
    if (!scratch) return SWIATTN_ECUDA;
    const int fit = decode_block_check(dtype, d, Hq, Hkv, false);
    if (fit != SWIATTN_OK) return fit;
    // Every chunk's partial is written before the combine reads it, so the
    // scratch needs no clearing between calls.
    return launched(launch_decode(q, k_cache, v_cache, seq_lens, gate, o, lse, B, Lmax, Hq, Hkv,
                                  d, W, 0, scale, dtype, L, reinterpret_cast<char*>(scratch),
                                  di.err, static_cast<cudaStream_t>(stream)));
}

size_t swiattn_decode_paged_workspace(int B, int max_pages, int page_size, int Hq, int Hkv, int d,
                                      int W, int n_anchor, int dtype) {
    if (page_size <= 0 || (page_size & (page_size - 1)) != 0 || max_pages <= 0) return 0;
    const int64_t max_len = (int64_t)max_pages * page_size;
    if (max_len > (1 << 30)) return 0;
    return swiattn_decode_anchored_workspace(B, (int)max_len, Hq, Hkv, d, W, n_anchor, dtype);
}

int swiattn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                         const int32_t* block_table, const int32_t* seq_lens, const uint8_t* gate,
                         void* o, float* lse, int B, int max_pages, int page_size, int num_pages,
                         int Hq, int Hkv, int d, int W, int n_anchor, float scale, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream) {
    if (page_size <= 0 || (page_size & (page_size - 1)) != 0 || max_pages <= 0 || num_pages <= 0)
        return SWIATTN_EINVAL;
    const int64_t max_len = (int64_t)max_pages * page_size;
    if (max_len > (1 << 30)) return SWIATTN_EINVAL;
    if (!block_table) return SWIATTN_EINVAL;
    const int st = decode_args_ok(q, k_pages, v_pages, seq_lens, gate, o, B, (int)max_len, Hq, Hkv,
                                  d, W, n_anchor, scale, dtype);
    if (st != SWIATTN_OK) return st;
    const DecodeWs L = decode_ws_layout(B, (int)max_len, Hq, d, n_anchor);
    if (!workspace || !aligned256(workspace) || workspace_bytes < L.total) return SWIATTN_EINVAL;
    DeviceInfo di;
    if (!device_info(di)) return SWIATTN_ECUDA;
    const int fit = decode_block_check(dtype, d, Hq, Hkv, true);
    if (fit != SWIATTN_OK) return fit;
    int lg = 0;
    while ((1 << lg) < page_size) ++lg;
    return launched(launch_decode_paged(q, k_pages, v_pages, block_table, seq_lens, gate, o, lse,
                                        B, max_pages, lg, num_pages, Hq, Hkv, d, W, n_anchor,
                                        scale, dtype, L, static_cast<char*>(workspace), di.err,
                                        static_cast<cudaStream_t>(stream)));
}

size_t swiattn_dual_branch_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype) {
    if (!attn_shape_ok(B, N, Hq, Hkv, d, W)) return 0;
    return dual_ws_layout(B, N, Hq, d, dtype).total;
}

int swiattn_dual_branch(const void* q, const void* k, const void* v, const float* logits,
                        const float* nll, void* o_full, void* o_swa, void* o_gated,
                        float* lse_gated, float* mse,
                        float* gamma, float* reg_loss, int B, int N, int Hq, int Hkv, int d, int W,
                        float scale, float gamma_base, float eps, float alpha, int dtype,
                        void* workspace, size_t workspace_bytes, void* stream) {
    if (!attn_shape_ok(B, N, Hq, Hkv, d, W)) return SWIATTN_EINVAL;
    if (!q || !k || !v || !logits || !nll || !o_full || !o_swa || !mse || !gamma || !reg_loss)
        return SWIATTN_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_full) ||
        !aligned16(o_swa) || (o_gated && !aligned16(o_gated)))
        return SWIATTN_EINVAL;
    if (!(scale > 0.f)) return SWIATTN_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SWIATTN_F32) {
        float* lf = nullptr;
        float* ls = nullptr;
        if (lse_gated) {   // both branches' lse go through the workspace
            const DualWs L = dual_ws_layout(B, N, Hq, d, dtype);
            if (!workspace || !aligned256(workspace) || workspace_bytes < L.total)
                return SWIATTN_EINVAL;
            lf = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.lse_full);
            ls = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.lse_swa);
        }
        cudaError_t e = launch_simt_attention(q, k, v, nullptr, 1, o_full, lf, B, N, Hq, Hkv, d, W,
                                              0, scale, dtype, s);
        if (e == cudaSuccess)
            e = launch_simt_attention(q, k, v, nullptr, 0, o_swa, ls, B, N, Hq, Hkv, d, W, 0,
                                      scale, dtype, s);
        if (e == cudaSuccess)
            e = launch_dual_epilogue_f32(static_cast<const float*>(o_full),
                                         static_cast<const float*>(o_swa), logits, nll,
                                         static_cast<float*>(o_gated), lf, ls, lse_gated, mse,
                                         gamma, reg_loss, B, N, Hq, d, gamma_base, eps, alpha, s);
        return launched(e);
    }
    if (dtype != SWIATTN_BF16) return SWIATTN_EINVAL;
    if (d != kHD) return SWIATTN_EUNSUPPORTED;
    const DualWs L = dual_ws_layout(B, N, Hq, d, dtype);
    if (!workspace || !aligned256(workspace) || workspace_bytes < L.total) return SWIATTN_EINVAL;
    DeviceInfo di;
    if (!device_info(di)) return SWIATTN_ECUDA;
    float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.mse_part);
    TcAttnArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k;
    a.v = v;
    a.logits = logits;
    a.o = o_full;
    a.o_swa = o_swa;
    a.o_gated = o_gated;
    a.lse = lse_gated;
    a.mse_part = part;
    a.snap = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.snap);
    a.counter = reinterpret_cast<int*>(static_cast<char*>(workspace) + L.counter);
    a.B = B;
    a.N = N;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.W = W;
    a.scale = scale;
    cudaError_t e = launch_dual_tc(a, di.err, di.sms, s);
    if (e == cudaSuccess)
        e = launch_dual_epilogue_parts(part, logits, nll, mse, gamma, reg_loss, B, N, Hq,
                                       gamma_base, eps, alpha, s);
    return launched(e);
}

size_t swiattn_prefill_backward_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype) {
    if (!attn_shape_ok(B, N, Hq, Hkv, d, W)) return 0;
    if (dtype != SWIATTN_BF16) {   // fp32 path: D per row
        const size_t n = sizeof(float) * (size_t)B * N * Hq;
        return (n + 255) & ~static_cast<size_t>(255);
    }
    return bwd_ws_layout(B, N, Hq, Hkv).total;
}

int swiattn_prefill_backward(const void* q, const void* k, const void* v, const uint8_t* gate,
                             const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                             void* dv, int B, int N, int Hq, int Hkv, int d, int W, float scale,
                             int dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (!attn_shape_ok(B, N, Hq, Hkv, d, W)) return SWIATTN_EINVAL;
    if (!q || !k || !v || !gate || !o || !lse || !d_o || !dq || !dk || !dv) return SWIATTN_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(d_o) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return SWIATTN_EINVAL;
    if (!(scale > 0.f)) return SWIATTN_EINVAL;
    if (dtype != SWIATTN_BF16 && dtype != SWIATTN_F32) return SWIATTN_EINVAL;
    if (dtype == SWIATTN_BF16 && d != kHD) return SWIATTN_EUNSUPPORTED;
    const size_t need = swiattn_prefill_backward_workspace(B, N, Hq, Hkv, d, W, dtype);
    if (!workspace || !aligned256(workspace) || workspace_bytes < need) return SWIATTN_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == SWIATTN_F32) {
        prof_start(s);
        cudaError_t e = launch_simt_backward(
            static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
            gate, static_cast<const float*>(o), lse, static_cast<const float*>(d_o),
            static_cast<float*>(dq), static_cast<float*>(dk), static_cast<float*>(dv), B, N, Hq, Hkv,
            d, W, scale, static_cast<float*>(workspace), s);
        prof_stop(s);
        return launched(e);
    }
    DeviceInfo di;
    if (!device_info(di)) return SWIATTN_ECUDA;
    const BwdWs L = bwd_ws_layout(B, N, Hq, Hkv);
    char* ws = static_cast<char*>(workspace);
    cudaError_t e = launch_bwd_schedule(gate, q, o, lse, d_o, B, N, Hq, Hkv, W, L, ws, di.sms, s);
    if (e != cudaSuccess) return SWIATTN_ECUDA;
    TcBwdArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k;
    a.v = v;
    a.d_o = d_o;
    a.gate = gate;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.L = &L;
    a.ws = ws;
    a.B = B;
    a.N = N;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.W = W;
    a.scale = scale;
    prof_start(s);
    e = launch_bwd_dkdv(a, di.err, di.sms, s);
    if (e == cudaSuccess) e = launch_bwd_dq(a, di.err, di.sms, s);
    prof_stop(s);
    return launched(e);
}

size_t swiattn_route_backward_workspace(int64_t tokens, int d_model, int dtype) {
    (void)dtype;
    if (tokens < 0 || d_model <= 0) return 0;
    const size_t n = sizeof(float) * (size_t)route_bwd_chunks(tokens) * (size_t)d_model;
    return (n + 255) & ~static_cast<size_t>(255);
}

int swiattn_route_backward(const void* h, const void* w, const float* logits, const void* o_full,
                           const void* o_swa, const void* d_o, const float* gamma,
                           const float* d_reg, int64_t tokens, int hd, int d_model, int dtype,
                           float* d_logits, void* dh, float* dw, float* db, void* workspace,
                           size_t workspace_bytes, void* stream) {
    if (tokens < 0 || hd <= 0) return SWIATTN_EINVAL;
    if (dtype != SWIATTN_BF16 && dtype != SWIATTN_F32) return SWIATTN_EINVAL;
    if (hd % 8 != 0) return SWIATTN_EINVAL;
    if ((dh || dw || db) && (d_model <= 0 || d_model % 8 != 0)) return SWIATTN_EINVAL;
    if (tokens == 0) return SWIATTN_OK;
    if (!logits || !o_full || !o_swa || !d_o || !d_logits || (d_reg && !gamma))
        return SWIATTN_EINVAL;
    if (!aligned16(o_full) || !aligned16(o_swa) || !aligned16(d_o)) return SWIATTN_EINVAL;
    if ((dh || dw) && (!h || !w || !aligned16(h) || !aligned16(w))) return SWIATTN_EINVAL;
    if ((dh && !aligned16(dh)) || (dw && !aligned16(dw))) return SWIATTN_EINVAL;
    if (dw) {
        const size_t need = swiattn_route_backward_workspace(tokens, d_model, dtype);
        if (!workspace || !aligned256(workspace) || workspace_bytes < need) return SWIATTN_EINVAL;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    prof_start(s);
    const cudaError_t e = launch_route_backward(h, w, logits, o_full, o_swa, d_o, gamma, d_reg,
                                                tokens, hd, d_model, dtype, d_logits, dh, dw, db,
                                                static_cast<float*>(workspace), s);
    prof_stop(s);
    return launched(e);
}

}  // extern "C"
