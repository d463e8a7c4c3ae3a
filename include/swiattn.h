/*
 * swiattn.h -- C ABI of libswiattn, the GB300 (sm_103a) hot path of SwiAttn,
 * token-level routed hybrid attention.
 *
 * The method (SwiAttn report, paper-daily.com retrieval report of 2026-03-31,
 * section 2 "方法详解"): at every layer a linear router R scores each token;
 * the hard gate sigma = 1(sigmoid(R(h)) > 0.5) chooses, per query row, causal
 * full attention over keys [0, i] (O_FULL) or sliding-window attention over
 * keys [i-W+1, i] (O_SWA, the window definition of the weimeta.cn glossary
 * "滑窗注意力 Sliding Window Attention 是什么", section "详细解释").  Both
 * branches share one Q/K/V and, at decode time, one KV cache; the layer output
 * is O = sigma*O_FULL + (1-sigma)*O_SWA.  Training adds the divergence
 * ||o_FULL - o_SWA||^2, the adaptive weight
 * gamma = gamma_base/(eps + NLL + alpha*||.||^2) and the regulariser
 * gamma*softplus(R(h)).
 *
 * Conventions for every call
 *  - Pointers are DEVICE pointers unless stated; the caller allocates and owns
 *    every buffer, including workspaces.  The library keeps no pointer after a
 *    call returns and allocates no device memory.
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream) and is asynchronous: a return of SWIATTN_OK
 *    means "validated and launched".
 *  - Arguments are validated before anything is launched; on any error
 *    nothing is launched and outputs are untouched.
 *  - Layouts are row-major and contiguous: q [B,N,Hq,d]; k, v [B,N,Hkv,d];
 *    decode caches [B,Lmax,Hkv,d]; per-token arrays [B,N].  Every tensor
 *    pointer must be 16-byte aligned.  Query head h reads KV head
 *    h / (Hq/Hkv) (contiguous GQA groups; the glossary's FAQ on GQA).
 *  - Rows are 0-based; the window is clipped at key 0.  The gate is
 *    logit > 0 (strictly), which is sigmoid(logit) > 0.5.
 *  - dtype selects the element type of the q/k/v/h/w/o tensors of the call:
 *    SWIATTN_BF16 (compute in fp32 with bf16 operands on the tensor cores) or
 *    SWIATTN_F32 (fp32 end to end on CUDA cores).  Statistics (logits, lse,
 *    mse, gamma, reg_loss, nll) are always fp32.
 *  - Device-side waits are bounded; if one ever expires the kernel returns
 *    early and records the fact, which swiattn_get_device_error reports.
 */
#ifndef SWIATTN_H
#define SWIATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SWIATTN_OK = 0,
    SWIATTN_EINVAL = 1,        /* bad pointer, size, alignment or workspace too small */
    SWIATTN_EUNSUPPORTED = 2,  /* valid request the library does not implement (e.g. d) */
    SWIATTN_ECUDA = 3,         /* a CUDA runtime/driver call failed (launch, symbol, map) */
    SWIATTN_ETIMEOUT = 4       /* a device-side bounded wait expired (from get_device_error) */
} swiattn_status;

typedef enum { SWIATTN_F32 = 0, SWIATTN_BF16 = 1 } swiattn_dtype;

/* Router GEMV and hard gate (report section 2, router design; one scalar per
 * token per layer, shared by every head):
 *   logits[t] = sum_j h[t,j] * w[j] + bias   (fp32 accumulation)
 *   gate[t]   = logits[t] > 0 ? 1 : 0
 * h [tokens, d_model], w [d_model] of `dtype`; logits fp32 [tokens];
 * gate uint8 [tokens].  d_model must be a multiple of 8 (bf16) or 4 (fp32).
 * tokens == 0 is a valid no-op. */
int swiattn_route(const void* h, const void* w, float bias, int64_t tokens, int d_model,
                  int dtype, float* logits, uint8_t* gate, void* stream);

/* Bytes of device workspace swiattn_prefill needs for these sizes. */
size_t swiattn_prefill_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype);

/* Routed causal prefill (report section 2, dual-branch computation, inference
 * form).  For each batch b, query head h and row i, with
 *   [lo, hi] = gate[b,i] ? [0, i] : [max(0, i-W+1), i]
 * o[b,i,h,:] = softmax_j(scale * q_i . k_j) v_j over j in [lo, hi], which equals
 * sigma*O_FULL + (1-sigma)*O_SWA with a 0/1 gate.  Window rows cost about W
 * keys, routed rows about i keys: masked and out-of-window key tiles are never
 * visited.  gate uint8 [B,N]; o [B,N,Hq,d] of `dtype`; lse (nullable) fp32
 * [B,N,Hq] receives ln sum_j exp(scale * q_i . k_j) over the visited keys.
 * d in {64, 128} for SWIATTN_F32; d == 128 for SWIATTN_BF16.
 * workspace: at least swiattn_prefill_workspace(...) bytes, 256-byte aligned;
 * it is scratch only (its contents need not be preserved between calls).
 * Calls that share one workspace must not overlap in time. */
int swiattn_prefill(const void* q, const void* k, const void* v, const uint8_t* gate, void* o,
                    float* lse, int B, int N, int Hq, int Hkv, int d, int W, float scale,
                    int dtype, void* workspace, size_t workspace_bytes, void* stream);

/* swiattn_prefill with global anchors (SWA glossary, "详细解释" platform note on
 * 全局锚点重注入 and "SWA 落地的四个常见坑" pitfall 1, fix 2: every query also
 * attends the first tokens, which the window never evicts; 256 there).  A
 * window row i visits [0, min(n_anchor, i-W+1)) together with
 * [max(0, i-W+1), i]; a routed row visits [0, i] as before.  n_anchor >= 0;
 * 0 is swiattn_prefill.  Other arguments, and the workspace
 * (swiattn_prefill_workspace bytes), as swiattn_prefill. */
int swiattn_prefill_anchored(const void* q, const void* k, const void* v, const uint8_t* gate,
                             void* o, float* lse, int B, int N, int Hq, int Hkv, int d, int W,
                             int n_anchor, float scale, int dtype, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Bytes of device workspace swiattn_prefill_host needs: device copies of q, k,
 * v, gate and o (and lse) plus the prefill's own workspace (0 for invalid sizes). */
size_t swiattn_prefill_host_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype);

/* swiattn_prefill_anchored from and to HOST memory, for callers that keep
 * tensors on the host: enqueues on `stream` the copies of q, k, v, gate to
 * device staging inside `workspace` (one cudaMemcpyAsync each), the prefill,
 * and the copies of o (and lse, when lse_host is not null) back to the host.
 * q_host, k_host, v_host, gate_host, o_host, lse_host are host pointers with
 * the layouts of swiattn_prefill; with page-locked (pinned) host memory every
 * copy is asynchronous, with pageable memory the CUDA runtime synchronises
 * around it.  The results are in o_host once the stream reaches the end of the
 * call.  workspace: device memory of at least swiattn_prefill_host_workspace
 * bytes, 256-byte aligned; other arguments as swiattn_prefill_anchored. */
int swiattn_prefill_host(const void* q_host, const void* k_host, const void* v_host,
                         const uint8_t* gate_host, void* o_host, float* lse_host, int B, int N,
                         int Hq, int Hkv, int d, int W, int n_anchor, float scale, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace swiattn_route_prefill needs (0 for invalid sizes). */
size_t swiattn_route_prefill_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype);

/* One layer's router and routed prefill in one call (report section 2: the
 * router's hard gate decides, per token, the key set of the prefill):
 *   logits[b*N+i] = h[b*N+i,:] . w + bias,  gate[b*N+i] = logits > 0,
 * then o = swiattn_prefill_anchored(q, k, v, gate, ...).  h [B*N, d_model]
 * and w [d_model] of `dtype` (16-byte aligned; d_model a multiple of 8 for
 * bf16, 4 for fp32); logits fp32 [B*N] and gate uint8 [B*N] are written (the
 * gates are the prefill's); the remaining arguments as
 * swiattn_prefill_anchored (n_anchor 0: no anchors).  For bf16 the router GEMV
 * and the prefill schedule are one launch (the CTA that finishes the GEMV last
 * plans the prefill over all gates), so the call is two kernel launches and a
 * 4-byte reset of a counter in the workspace.  Results equal those of
 * swiattn_route followed by swiattn_prefill_anchored bit for bit.
 * workspace: at least swiattn_route_prefill_workspace(...) bytes, 256-byte
 * aligned, scratch only; calls that share one must not overlap in time. */
int swiattn_route_prefill(const void* h, const void* w, float bias, int d_model, const void* q,
                          const void* k, const void* v, void* o, float* lse, float* logits,
                          uint8_t* gate, int B, int N, int Hq, int Hkv, int d, int W, int n_anchor,
                          float scale, int dtype, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Bytes of device workspace swiattn_decode needs for these sizes. */
size_t swiattn_decode_workspace(int B, int Lmax, int Hq, int Hkv, int d, int W, int dtype);

/* One decode step over a shared KV cache (report section 2: both branches
 * share the cache; section 6: decode reads the last W entries or all of them).
 * Sequence b holds seq_lens[b] tokens (1 <= seq_lens[b] <= Lmax), the newest
 * being the query's own, at position L = seq_lens[b]-1.  The query reads cache
 * entries [max(0, L-W+1), L] if gate[b] == 0, else [0, L].
 * q [B,Hq,d]; k_cache, v_cache [B,Lmax,Hkv,d]; seq_lens int32 [B];
 * gate uint8 [B]; o [B,Hq,d]; lse (nullable) fp32 [B,Hq].  A seq_lens[b]
 * outside [1, Lmax] (a device-resident input) is clamped into it and
 * swiattn_get_device_error then reports SWIATTN_EINVAL.
 * d in {64, 128}; Hq/Hkv in {1, 2, 4, 8}; Lmax <= 2^30 (larger:
 * SWIATTN_EUNSUPPORTED).  One thread per 16 bytes of a
 * token row (Hkv*d/8 threads for bf16, Hkv*d/4 for fp32, rounded up to 32)
 * must fit one block of the split kernel on the device: at most 1024 threads,
 * fewer where the kernel's register use takes more (e.g. 896 for bf16, d=128,
 * Hq = Hkv; 256 for Hq = 8*Hkv).  A larger request returns
 * SWIATTN_EUNSUPPORTED and launches nothing; so do swiattn_decode_anchored,
 * swiattn_decode_paged and swiattn_decode_noalloc, whose limits are these.
 * workspace: at least swiattn_decode_workspace(...) bytes, scratch only; for
 * B <= 32 the call first clears a 4-byte chunk counter in it on `stream`
 * (cudaMemsetAsync), then launches its two kernels there. */
int swiattn_decode(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* seq_lens, const uint8_t* gate, void* o, float* lse, int B,
                   int Lmax, int Hq, int Hkv, int d, int W, float scale, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace swiattn_decode_anchored needs (0 for invalid sizes). */
size_t swiattn_decode_anchored_workspace(int B, int Lmax, int Hq, int Hkv, int d, int W,
                                         int n_anchor, int dtype);

/* swiattn_decode with global anchors (SWA glossary, "详细解释" platform note on
 * 全局锚点重注入 and "SWA 落地的四个常见坑" pitfall 1, fix 2: the first tokens'
 * K/V stay in the cache and every query also attends them).  A window query
 * at position L-1 reads cache entries [0, min(n_anchor, L)) together with
 * [max(0, L-W), L-1]; a routed query reads [0, L-1] as before.  n_anchor >= 0;
 * 0 is swiattn_decode.  Other arguments as swiattn_decode.
 * workspace: at least swiattn_decode_anchored_workspace(...) bytes. */
int swiattn_decode_anchored(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* seq_lens, const uint8_t* gate, void* o, float* lse,
                            int B, int Lmax, int Hq, int Hkv, int d, int W, int n_anchor,
                            float scale, int dtype, void* workspace, size_t workspace_bytes,
                            void* stream);

/* swiattn_decode without a workspace argument, for callers that cannot
 * allocate device memory (for example code that runs inside an allocator-free
 * runtime or a host framework that owns every device allocation and exposes
 * none to plug-ins).  The paper has no counterpart: this is a deployment
 * convenience.  Arguments, layouts, results and the device-side report of a
 * seq_lens[b] outside [1, Lmax] (clamped, then SWIATTN_EINVAL from
 * swiattn_get_device_error) are those of swiattn_decode.
 *  - The split-KV partials go to one fixed 16 MiB device array inside the
 *    library, which every GPU that loads the library holds until the process
 *    exits.  A call whose partials, B * max(17, ceil(Lmax/256) + 1) * Hq *
 *    (d+2) * 4 bytes rounded up to 256, plus 256 bytes, exceed 16 MiB returns
 *    SWIATTN_EINVAL and launches nothing (e.g. B=16, Hq=16, d=128 allows Lmax
 *    up to 32 000).
 *  - The call allocates nothing.  Its first call on a device looks up that
 *    array's device address (once per device, with the device current); make
 *    that first call before any stream capture.
 *  - All calls share the one array: calls that overlap on the GPU (different
 *    streams, or different host threads without ordering) race and corrupt
 *    each other's results.  No state carries over between calls that do not
 *    overlap. */
int swiattn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, const uint8_t* gate, void* o, float* lse,
                           int B, int Lmax, int Hq, int Hkv, int d, int W, float scale, int dtype,
                           void* stream);

/* Bytes of device workspace swiattn_decode_paged needs for these sizes
 * (0 for invalid sizes). */
size_t swiattn_decode_paged_workspace(int B, int max_pages, int page_size, int Hq, int Hkv, int d,
                                      int W, int n_anchor, int dtype);

/* swiattn_decode over a paged KV cache (a serving cache layout; the report's
 * decode, section 2 and 6, reads the last W or all cache entries of each
 * sequence, whatever their placement).  Token t of sequence b is row
 * t % page_size of physical page block_table[b * max_pages + t / page_size]
 * of the pool k_pages, v_pages [num_pages, page_size, Hkv, d].
 * page_size is a power of two; seq_lens[b] <= max_pages * page_size.  The
 * block table and seq_lens are device arrays: a table entry the call reads
 * that lies outside [0, num_pages) is read as page 0, and a seq_lens[b]
 * outside [1, max_pages * page_size] is clamped into it; either way
 * swiattn_get_device_error then reports SWIATTN_EINVAL (no out-of-range read
 * is made).  Entries of pages a call does not visit are not read.  Other arguments, layouts
 * and results are those of swiattn_decode_anchored (n_anchor = 0: of
 * swiattn_decode).  A batched step over several
 * layers is one call with (layer, sequence) flattened into B (one pool, or
 * per-layer pools laid end to end with the table entries offset).
 * workspace: at least swiattn_decode_paged_workspace(...) bytes. */
int swiattn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                         const int32_t* block_table, const int32_t* seq_lens, const uint8_t* gate,
                         void* o, float* lse, int B, int max_pages, int page_size, int num_pages,
                         int Hq, int Hkv, int d, int W, int n_anchor, float scale, int dtype,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace swiattn_dual_branch needs for these sizes. */
size_t swiattn_dual_branch_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype);

/* Training-side dual-branch forward (report section 2, dual-branch computation
 * and adaptive regularisation loss).  For every token both branches:
 *   o_full[b,i,h,:] over keys [0, i];  o_swa[b,i,h,:] over [max(0,i-W+1), i]
 *   mse[b,i]      = sum_{h,c} (o_full - o_swa)^2, from the fp32 values before
 *                   any rounding to the output type
 *   gamma[b,i]    = gamma_base / (eps + nll[b,i] + alpha * mse[b,i])
 *   reg_loss[b,i] = gamma[b,i] * softplus(logits[b,i])
 *   o_gated[b,i,h,:] (nullable) = logits[b,i] > 0 ? o_full : o_swa
 *   lse_gated[b,i,h] (nullable) = the log-sum-exp of the branch o_gated took
 *                   (what swiattn_prefill_backward needs with o_gated)
 * logits, nll fp32 [B,N] (nll is treated as a constant input); o_full, o_swa,
 * o_gated [B,N,Hq,d] of `dtype`; lse_gated fp32 [B,N,Hq]; mse, gamma, reg_loss
 * fp32 [B,N].
 * The report's values are gamma_base = 1e-3, eps = 0.1, alpha = 100.
 * workspace: at least swiattn_dual_branch_workspace(...) bytes, scratch only. */
int swiattn_dual_branch(const void* q, const void* k, const void* v, const float* logits,
                        const float* nll, void* o_full, void* o_swa, void* o_gated,
                        float* lse_gated, float* mse, float* gamma, float* reg_loss, int B, int N,
                        int Hq, int Hkv, int d, int W, float scale, float gamma_base, float eps,
                        float alpha, int dtype, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Bytes of device workspace swiattn_prefill_backward needs for these sizes. */
size_t swiattn_prefill_backward_workspace(int B, int N, int Hq, int Hkv, int d, int W, int dtype);

/* Gradient of swiattn_prefill for training (report section 2, router design:
 * the straight-through gate's forward value is the hard 0/1, so the output
 * gradient of row i reaches only the branch its gate selected).  Inputs: the
 * forward's q, k, v, gate, its output o and lse (swiattn_prefill with
 * lse != NULL; the same values the dual branch's gated output has), and
 * d_o = dLoss/do [B,N,Hq,d].  Outputs dq [B,N,Hq,d] and dk, dv [B,N,Hkv,d] of
 * `dtype`, by the chain rule through each row's softmax over its visited keys
 * [lo, hi] (as in swiattn_prefill):
 *   D_i = <d_o_i, o_i>,   p_ij = exp(scale q_i.k_j - lse_i),
 *   dS_ij = p_ij (<d_o_i, v_j> - D_i),
 *   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,
 *   dv_j = sum_i p_ij d_o_i,
 * the sums running over the (i, j) pairs the forward visits; dk and dv sum
 * over the query heads of each GQA group.  Every element of dq, dk, dv is
 * written.  No atomics: results are bitwise repeatable.  Support as for
 * swiattn_prefill (bf16: d == 128, tensor cores; fp32: d in {64, 128}).
 * workspace: at least swiattn_prefill_backward_workspace(...) bytes, 256-byte
 * aligned, scratch only. */
int swiattn_prefill_backward(const void* q, const void* k, const void* v, const uint8_t* gate,
                             const void* o, const float* lse, const void* d_o, void* dq, void* dk,
                             void* dv, int B, int N, int Hq, int Hkv, int d, int W, float scale,
                             int dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace swiattn_route_backward needs (only when dw is
 * requested). */
size_t swiattn_route_backward_workspace(int64_t tokens, int d_model, int dtype);

/* Router backward through the straight-through gate and the adaptive
 * regulariser (report section 2).  The gate sigma = 1(s > 0.5) + s - sg(s),
 * s = sigmoid(logit), passes d sigma / d logit = s (1 - s); the output
 * O = sigma O_FULL + (1 - sigma) O_SWA gives dO / d sigma = O_FULL - O_SWA;
 * gamma is a coefficient of the regulariser (no gradient flows through it,
 * as through NLL).  Per token t:
 *   d_logits[t] = s_t (1 - s_t) * sum_c d_o[t,c] (o_full[t,c] - o_swa[t,c])
 *               + d_reg[t] * gamma[t] * s_t
 * with d_reg = dLoss/dreg_loss (nullable: no regulariser term).  Then through
 * the linear router logits = h.w + bias:
 *   dh[t,:] = d_logits[t] w,   dw = sum_t d_logits[t] h[t,:],   db = sum_t d_logits[t].
 * o_full, o_swa, d_o [tokens, hd] of `dtype` (hd = Hq*d: one token's attention
 * outputs); logits, gamma, d_reg fp32 [tokens]; h [tokens, d_model] and
 * w [d_model] of `dtype`; outputs d_logits fp32 [tokens], dh [tokens, d_model]
 * of `dtype`, dw fp32 [d_model], db fp32 [1].  dh, dw and db are each
 * nullable; h and w may be NULL when dh and dw both are.  hd and d_model are
 * multiples of 8.  dw and db are reduced in a fixed order (repeatable).
 * workspace: swiattn_route_backward_workspace(...) bytes when dw != NULL,
 * otherwise unused (may be NULL).  tokens == 0 is a valid no-op. */
int swiattn_route_backward(const void* h, const void* w, const float* logits, const void* o_full,
                           const void* o_swa, const void* d_o, const float* gamma,
                           const float* d_reg, int64_t tokens, int hd, int d_model, int dtype,
                           float* d_logits, void* dh, float* dw, float* db, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Synchronises `stream`, then returns and clears the device error word of the
 * current device: SWIATTN_OK, SWIATTN_ETIMEOUT if a bounded device wait
 * expired since the last query, or SWIATTN_ECUDA if the synchronisation itself
 * failed or a kernel found its shared memory not laid out as it requires (it
 * then returned without computing), or SWIATTN_EINVAL if a kernel met an
 * out-of-range device-resident input (e.g. a paged-decode block table entry). */
int swiattn_get_device_error(void* stream);

/* Static, NUL-terminated name of a status code. */
const char* swiattn_status_string(int status);

/* Timing hook.  When both are non-NULL, every later swiattn_prefill,
 * swiattn_decode, swiattn_dual_branch, swiattn_prefill_backward, swiattn_route
 * and swiattn_route_backward call records `start` (a cudaEvent_t passed as
 * void*) on its stream immediately before launching its dominant kernel (the
 * attention kernel, the decode split kernel, the backward's two attention
 * kernels, dK/dV then dQ, the router GEMV, or the router backward's three
 * kernels) and `stop` immediately after it, so cudaEventElapsedTime gives that
 * kernel's device time alone.  Passing NULL, NULL turns the hook off.  Process-wide setting;
 * the events stay owned by the caller and must outlive their use. */
void swiattn_set_profile_events(void* start, void* stop);

/* Number of SMs of the current device (the persistent kernels launch one CTA
 * per SM), or -1 on a CUDA error. */
int swiattn_num_sms(void);

/* Failure-detection aid with no counterpart in the paper: sets, on the
 * current device, how long a device-side wait of the tensor-core kernels
 * (routed prefill, dual branch, backward) may last before the kernel gives up,
 * records SWIATTN_ETIMEOUT for swiattn_get_device_error and returns early
 * without computing the rest of its work; ns = 0 restores the default of 2 s.
 * A tiny limit lets a test make such a wait run out on purpose and check that
 * the kernel stops cleanly (it still waits, with a separate fixed bound, for
 * its own copies and tensor-core operations in flight before it exits) and
 * that the next call computes normally.  Outputs of a call that timed out are
 * unspecified.  Synchronous; call it with no kernel of this library running. */
int swiattn_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* SWIATTN_H */
