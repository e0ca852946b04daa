/*
 * kvo.h -- C ABI of the GB300 sparse offloaded-KV decode step.
 *
 * One decode step per layer, as described in "DualDecoder: Accelerate Long
 * Context LLM Inference by Predictive Prefetch" (arXiv 2607.26475):
 *   1. select_topk       -- score every host-resident block against static
 *                           GPU-resident K landmarks and keep the exact top-k
 *                           (the retrieval index, §4.1, Fig. 6, Fig. 8), for the
 *                           true query and optionally a speculative one;
 *   2. index_diff        -- compare the true index with the predicted one: the
 *                           misses go to the urgent stream (§5.2, Fig. 10);
 *   3. gather_coalesced  -- coalesce an ascending index list into runs of
 *                           adjacent blocks and copy them host -> HBM into one
 *                           half of a two-layer ping-pong buffer (§5.4, Fig. 11;
 *                           "PulseInfer and the I/O Problem Behind Long-Context
 *                           Decoding" §2: gather-scatter coalescing of
 *                           fragmented transfers);
 *   4. sparse_decode_attn -- GQA decode attention over the gathered blocks and
 *                           over a GPU-resident recent window, the two parts
 *                           fused by log-sum-exp ("Scaling Attention Beyond GPUs
 *                           for LLM Inference", abstract); merge_lse exposes
 *                           the fusion on its own.
 * kvo_decode_step runs all four for every layer with the stream/event schedule
 * of §5.3-§5.4 (prefetch for layer l+2 after layer l's attention).
 *
 * Conventions
 *  - Every call returns kvo_status and never aborts, traps or exits.  Host-side
 *    argument checks come first; on failure nothing is launched and
 *    kvo_last_error() describes the problem.  Errors the GPU detects (an index
 *    out of range in a caller-supplied list) are recorded in a device status
 *    word read by kvo_device_status().
 *  - All device work is enqueued on the caller's stream (a cudaStream_t passed
 *    as void*) and is asynchronous.  NULL selects the context's own compute
 *    stream (for gather_coalesced: its prefetch or urgent stream), which does
 *    not synchronize with the legacy default stream; pass cudaStreamLegacy
 *    ((void*)0x1) to order a call on the legacy default stream.
 *  - bf16 = IEEE bfloat16 bit patterns (uint16).  Sizes are element counts.
 *  - Notation: b batch, Hq / Hkv query / KV heads, r = Hq / Hkv, d head dim,
 *    B block size (tokens), k top-k, W window, len_b context of request b,
 *    C_b = (len_b - W) / B host-resident candidate blocks, G = b * Hkv groups.
 *    KV head g serves query heads g*r .. g*r + r - 1.
 *  - No CPU fallback exists: without a CUDA device the calls fail with
 *    KVO_ERR_CUDA.
 *  - Concurrency on one context.  The context owns scratch that some calls
 *    use while their kernels run; two calls using the same scratch must not
 *    overlap on the GPU (issue them on one stream, or order them with events),
 *    or their results are undefined.  The scratch classes:
 *      [sel]  selection keys, histograms and tickets: select_topk;
 *      [att]  attention work items, partial results and tickets:
 *             sparse_decode_attn, sparse_decode_attn_cobatch;
 *      [runs] the run list of gather_coalesced when runs_out is NULL (one per
 *             value of `urgent`);
 *      [buf]  the ping-pong halves / resident sets: gather_coalesced writes the
 *             slots it is given, the attention calls read the slots named by
 *             slot_of_true -- a slot must not be written while it is read;
 *      [all]  kvo_decode_step, kvo_decode_step_dual and kvo_append use every
 *             class (and the step state, window and landmarks): nothing else
 *             may overlap them on the same context.
 *    Calls of different classes may overlap freely (e.g. select_topk of layer
 *    l + 1 on one stream beside sparse_decode_attn of layer l on another).
 *    index_diff uses no context scratch (only its own outputs); merge_lse,
 *    kvo_plan_select and kvo_plan_attention need no context.  The device status word is updated
 *    atomically and may be written by overlapping calls.  Host-side calls that
 *    change settings (kvo_set_*, kvo_reset_prediction, kvo_profile*) first
 *    synchronize the context's own streams but not the caller's: make sure no
 *    call of this context is in flight on other streams.  Distinct contexts
 *    share nothing.
 */
#ifndef KVO_H
#define KVO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVO_OK = 0,
    KVO_ERR_INVALID = 1,   /* bad argument (null pointer, out-of-range size, bad config) */
    KVO_ERR_CUDA = 2,      /* a CUDA runtime call failed (see kvo_last_error) */
    KVO_ERR_OOM = 3,       /* device allocation failed */
    KVO_ERR_TIMEOUT = 4,   /* a bounded device wait gave up */
    KVO_ERR_STATE = 5,     /* call not valid in the context's current state */
    KVO_ERR_DEVICE = 6     /* the device status word holds an error */
} kvo_status;

/* device status word bits (kvo_device_status) */
#define KVO_DEV_BAD_BLOCK_ID 0x1   /* a block id >= C_b or < 0 in an index list */
#define KVO_DEV_BAD_SLOT     0x2   /* a slot >= 2k or a run past the buffer */
#define KVO_DEV_BAD_COUNT    0x4   /* a count outside [0, k] */
#define KVO_DEV_UNSORTED     0x8   /* an index list that is not strictly ascending */
#define KVO_DEV_TIMEOUT      0x10  /* a bounded device wait gave up */

typedef void* kvo_stream_t;        /* cudaStream_t */
typedef struct kvo_ctx kvo_ctx;    /* opaque, owned by the library */

typedef struct {
    int32_t batch;        /* b >= 1 */
    int32_t n_q_heads;    /* Hq, a multiple of Hkv, r = Hq / Hkv <= 16 */
    int32_t n_kv_heads;   /* Hkv >= 1 */
    int32_t head_dim;     /* d: 64 or 128 */
    int32_t block_size;   /* B >= 1 tokens per landmark block */
    int32_t top_k;        /* k >= 1, k <= C_b for every request */
    int32_t window;       /* W >= 0 recent tokens kept on the GPU */
    int32_t n_layers;     /* >= 1 */
    const int32_t* seq_lens; /* host [b]; len_b >= W, (len_b - W) % B == 0 */
    int32_t max_append;   /* tokens each request may grow by through kvo_append (0: fixed cache).
                             > 0 needs W > 0 and W % B == 0; the host arrays then reserve
                             len_b + max_append rows per (request, KV head). */
    int32_t resident;     /* 0: two-layer ping-pong buffer (DualDecoder §5.4).  1: cross-step delta
                             prefetch -- every layer keeps a GPU-resident set of 2k block slots per
                             (request, KV head) across decode steps, and kvo_decode_step fetches
                             only the blocks the set lacks (see kvo_resident_slots). */
} kvo_config;

/*
 * kv_offload_init -- build a context for one KV cache.
 *   k_host[l], v_host[l]: page-locked host memory that the device can address
 *       (cudaHostAlloc / torch pin_memory, or cudaHostRegister'ed), one per
 *       layer, packed request after request as [b][Hkv][cap_b][d] bf16 with
 *       cap_b = len_b + max_append (request b starts at element
 *       (sum_{b'<b} cap_b') * Hkv * d; rows >= len_b are spare capacity that
 *       kvo_append fills).  Caller-owned; must stay valid and unchanged (apart
 *       from what kvo_append writes) until kv_offload_destroy.
 *   k_win[l], v_win[l]: device memory [b][Hkv][W][d] bf16 holding tokens
 *       [len_b - W, len_b) of each request (the recent window).  Caller-owned;
 *       with max_append > 0 they are copied into the library's window ring at
 *       init and not read again.
 *   On success *out owns: the K landmarks of every layer (fp32 block means,
 *   or the bf16 key itself when B == 1; DualDecoder §4.1, Fig. 8), built here
 *   synchronously from k_host; the two ping-pong halves of K and V
 *   ([2][G][2k][B][d] bf16: slots [0,k) take prefetched blocks, [k,2k) misses);
 *   scratch; and three streams: compute, prefetch (lowest priority) and
 *   urgent (highest priority; DualDecoder Fig. 10).  With resident = 1 it also
 *   owns one resident set per layer ([G][2k][B][d] K and V each), its slot
 *   table and block map (see kvo_resident_slots).
 *   Errors: KVO_ERR_INVALID (config or pointers), KVO_ERR_OOM, KVO_ERR_CUDA.
 */
kvo_status kv_offload_init(const kvo_config* cfg, void* const* k_host, void* const* v_host,
                           const void* const* k_win, const void* const* v_win, kvo_ctx** out);

/* kv_offload_destroy -- synchronize and free everything the context owns. NULL is a no-op. */
kvo_status kv_offload_destroy(kvo_ctx* ctx);

/*
 * select_topk -- retrieval index of one layer (DualDecoder §4.1, Fig. 6).
 *   q, q_spec: device [b][Hq][d] bf16; q_spec may be NULL.
 *   Score of block j of group (b, g): s_j = sum_{h in group g} q_h . L_j
 *   (fp32).  idx_true[G][k] (device int32) receives the k highest-scoring
 *   blocks in ascending id order, ties to the lower id.  When q_spec is given,
 *   idx_pred[G][k] receives the same for q_spec from the same landmark pass
 *   (the speculative look-ahead query of the dual-token scheme, §5.2).
 *   Launched as a programmatic dependent of the kernel before it on `stream`:
 *   it reads nothing before that kernel has completed (stream order holds);
 *   only its launch overlaps that kernel's tail.
 *   Concurrency: [sel] -- one select_topk at a time per context.
 */
kvo_status select_topk(kvo_ctx* ctx, int layer, const void* q, const void* q_spec,
                       int32_t* idx_true, int32_t* idx_pred, kvo_stream_t stream);

/*
 * index_diff -- predicted-vs-needed diff (DualDecoder §5.2, Fig. 10, Fig. 18).
 *   idx_true[G][k], idx_pred[G][k]: device int32, ascending per group;
 *   idx_pred NULL means nothing was predicted (every block is a miss).
 *   Outputs (device int32): miss_idx[G][k] = idx_true minus idx_pred ascending
 *   (first miss_cnt[g] entries valid), miss_cnt[G], slot_of_true[G][k]:
 *   the ping-pong slot holding idx_true[g][i] -- its position in idx_pred if
 *   predicted, else k + its rank among the misses.
 *   Concurrency: uses no context scratch; may overlap any call.
 */
kvo_status index_diff(kvo_ctx* ctx, const int32_t* idx_true, const int32_t* idx_pred,
                      int32_t* miss_idx, int32_t* miss_cnt, int32_t* slot_of_true,
                      kvo_stream_t stream);

/*
 * gather_coalesced -- coalesced host -> HBM gather into a ping-pong half
 *   (PulseInfer §2; DualDecoder §5.4, Fig. 11, Fig. 19).
 *   idx[G][k]: device int32 ascending block ids; cnt[G] valid entries per group
 *   (NULL: k each).  Each maximal run of adjacent ids becomes one copy of
 *   n_blocks * B * d bf16 of K and of V from layer `layer`'s host cache into
 *   buffer half `buf` (0|1), slots slot_base + i.. (slot_base 0 for the
 *   prefetched prediction, k for urgent misses).  runs_out (device int32
 *   [G][k][4] = {first block, n blocks, first slot, 0}) and n_runs_out
 *   (device int32 [G]) are optional.  `urgent` is informational for stream
 *   choice when stream is NULL: 1 = the urgent stream, 0 = the prefetch
 *   stream; the caller orders other work after it with events.
 *   Concurrency: [buf] (the slots written) and, with runs_out NULL, [runs] of
 *   its `urgent` value; gathers into disjoint slots with caller-owned run
 *   lists (or different `urgent` values) may overlap.
 */
kvo_status gather_coalesced(kvo_ctx* ctx, int layer, int buf, const int32_t* idx,
                            const int32_t* cnt, int slot_base, int urgent, int32_t* runs_out,
                            int32_t* n_runs_out, kvo_stream_t stream);

/*
 * sparse_decode_attn -- GQA decode attention of one layer.
 *   q: device [b][Hq][d] bf16.  slot_of_true: device [G][k] int32 (from
 *   index_diff).  Keys/values: the B tokens of every slot named in
 *   slot_of_true of buffer half `buf`, plus the W window tokens of layer
 *   `layer`.  Softmax scale 1/sqrt(d), natural-log lse, fp32 accumulate.
 *   fuse_window_merge = 1: o[b][Hq][d], lse[b][Hq] (fp32, device) hold the
 *   window and sparse parts fused by log-sum-exp.  fuse_window_merge = 0:
 *   o[2][b][Hq][d], lse[2][b][Hq]: part 0 sparse, part 1 window (an empty
 *   part has lse = -inf, o = 0).
 *   With the group-split kernel (kvo_set_attn_impl 2) the launch is a
 *   programmatic dependent of the kernel before it on `stream`, reading
 *   nothing before that kernel has completed.
 *   Concurrency: [att], and it reads [buf] -- one attention call at a time
 *   per context, with no write to the slots it reads in flight.
 */
kvo_status sparse_decode_attn(kvo_ctx* ctx, int layer, int buf, const void* q,
                              const int32_t* slot_of_true, float* o, float* lse,
                              int fuse_window_merge, kvo_stream_t stream);

/*
 * sparse_decode_attn_cobatch -- co-batched attention of the true and the
 * speculative query (DualDecoder §5.2, Fig. 18: the real and the speculative
 * token attend in one batched pass).  Both queries of a KV group attend, in
 * one kernel pass over the same K/V bytes, to the blocks named by
 * slot_of_true plus the window; the speculative query's r rows fill M rows
 * r..2r-1 of the tensor-core tiles, so 2r <= 16 is required.
 *   q, q_spec: device [b][Hq][d] bf16.  o, lse as in sparse_decode_attn;
 *   o_spec, lse_spec: the same layouts for the speculative query.
 *   Concurrency: as sparse_decode_attn ([att], reads [buf]).
 */
kvo_status sparse_decode_attn_cobatch(kvo_ctx* ctx, int layer, int buf, const void* q, const void* q_spec,
                                      const int32_t* slot_of_true, float* o, float* lse, float* o_spec,
                                      float* lse_spec, int fuse_window_merge, kvo_stream_t stream);

/*
 * merge_lse -- fuse two attention parts over disjoint key sets
 *   ("Scaling Attention Beyond GPUs for LLM Inference", abstract):
 *   M = max(lse1, lse2), w_i = exp(lse_i - M), o = (w1 o1 + w2 o2) / (w1 + w2),
 *   lse = M + ln(w1 + w2); two empty parts (-inf) give o = 0, lse = -inf.
 *   All pointers device fp32: o*[rows][d], lse*[rows].  o may alias o1 or o2;
 *   lse must not alias lse1 or lse2.
 *   No context needed.
 */
kvo_status merge_lse(const float* o1, const float* lse1, const float* o2, const float* lse2,
                     float* o, float* lse, int rows, int d, kvo_stream_t stream);

/*
 * kvo_decode_step -- one whole decode step over every layer, pipelined.
 *   q, q_spec: device [n_layers][b][Hq][d] bf16 (q_spec may be NULL: the
 *   prediction for the next step is then the true index of this step).
 *   o: device [n_layers][b][Hq][d] fp32, lse: [n_layers][b][Hq] fp32.
 *   Per layer l: select (true + speculative) -> diff against the prediction
 *   kept from the previous step -> urgent gather of the misses -> attention;
 *   the prefetch of layer l+2's prediction is issued on the prefetch stream
 *   once layer l's attention has released its ping-pong half.  The first
 *   step after init has no prediction, so every block is a miss.  All work is
 *   ordered after `stream`, and `stream` waits for the outputs; the prefetches
 *   this step issues for the next step may still be in flight on return (the
 *   next step orders itself after them; kvo_device_status, kvo_reset_prediction
 *   and kv_offload_destroy synchronize them).  With resident = 1 the step
 *   keeps per-layer resident sets and fetches only their delta instead (see
 *   kvo_resident_slots); layers given low-rank factors rebuild their missed
 *   keys on the GPU (kvo_set_lowrank_keys).
 *   Concurrency: [all] -- no other call on this context may overlap a step
 *   (the in-flight prefetches it leaves are ordered by the library itself).
 */
kvo_status kvo_decode_step(kvo_ctx* ctx, const void* q, const void* q_spec, float* o,
                           float* lse, kvo_stream_t stream);

/*
 * kvo_decode_step_dual -- kvo_decode_step whose attention is co-batched: each
 * layer's attention pass also produces the speculative query's output over the
 * same key set (o_spec [n_layers][b][Hq][d], lse_spec [n_layers][b][Hq] fp32),
 * as the dual-token pipeline needs it (DualDecoder §5.2).  q_spec is required;
 * 2r <= 16.
 */
kvo_status kvo_decode_step_dual(kvo_ctx* ctx, const void* q, const void* q_spec, float* o, float* lse,
                                float* o_spec, float* lse_spec, kvo_stream_t stream);

/*
 * kvo_set_graphs -- 1: warm decode steps (every step after the first) are
 * captured once per step parity into a CUDA graph and replayed, which removes
 * the host launch work and shortens the gaps between dependent kernels; a
 * graph is re-captured when the q/o/lse pointers of the call change or a
 * gather tuning call is made.  Profiling (kvo_profile) bypasses the graphs.
 * With resident = 1 only chain steps are replayed: no q_spec, no prefetch of
 * an earlier step still in flight and no layer with low-rank keys (their
 * kernels run one after another on the compute stream); other resident steps
 * are launched stream by stream.
 * 0 (default): every step is launched stream by stream.
 */
kvo_status kvo_set_graphs(kvo_ctx* ctx, int enable);

/*
 * kvo_append -- grow every request by one decode token (needs max_append > 0).
 *   k_new, v_new: device [n_layers][b][Hkv][d] bf16, the new token's key and
 *   value per layer and KV head.  The token joins the GPU-resident recent
 *   window (a library-owned ring of W + B tokens per layer and group, filled
 *   from k_win / v_win at init).  When the window reaches W + B tokens its
 *   oldest block leaves it: the B rows are written to the host cache (rows
 *   C_b*B .. of the group) and the block's landmark (mean key; the key itself
 *   for B == 1) becomes candidate block C_b, so C_b grows by one.  The
 *   attended set of later calls is the candidates' top-k plus the whole
 *   window (W to W + B - 1 tokens).  Ordered on `stream` like the other calls.
 *   Errors: KVO_ERR_STATE when the context was built with max_append == 0 or
 *   the reserved capacity is used up.
 *   Concurrency: [all].
 */
kvo_status kvo_append(kvo_ctx* ctx, const void* k_new, const void* v_new, kvo_stream_t stream);

/* Forget the predictions kept for the next step (next step starts cold). */
kvo_status kvo_reset_prediction(kvo_ctx* ctx);

/* kvo_get_stream -- which 0: compute, 1: prefetch, 2: urgent. */
kvo_status kvo_get_stream(kvo_ctx* ctx, int which, kvo_stream_t* out);

/*
 * kvo_device_status -- synchronize the context's streams and `stream`, return
 * and clear the device status word (KVO_DEV_* bits) in *code_out.
 * Returns KVO_ERR_DEVICE when it was nonzero.
 */
kvo_status kvo_device_status(kvo_ctx* ctx, int32_t* code_out, kvo_stream_t stream);

/*
 * Inspection, for tests and tools.
 *   kvo_landmarks: copy layer `layer`'s landmarks, in logical layout
 *   [G][C_max][d], to device memory `dst` (fp32 when B > 1; bf16 when B == 1),
 *   C_max = max_b C_b; rows past C_b are zero.
 *   kvo_buffer: device pointers of ping-pong half `buf` (0, 1) or, with
 *   resident = 1, of layer l's resident block set (buf = 2 + l), K and V, each
 *   [G][2k][B][d] bf16 (valid until destroy).  gather_coalesced,
 *   sparse_decode_attn and sparse_decode_attn_cobatch accept the same ids.
 *   kvo_info: sizes the context derived: [0] C_max, [1] landmark bytes per
 *   layer, [2] ping-pong bytes (both halves, K+V), [3] scratch bytes.
 */
kvo_status kvo_landmarks(kvo_ctx* ctx, int layer, void* dst, kvo_stream_t stream);
kvo_status kvo_buffer(kvo_ctx* ctx, int buf, void** k_out, void** v_out);

/*
 * Cross-step delta prefetch (resident = 1; "NeuroPrefetcher: Storage-Aware
 * Sparse LLM Inference via Delta Prefetching", title; DualDecoder §5.2 /
 * Fig. 18).  Per layer and (request, KV head) a table of 2k slots names the
 * block each slot of the layer's resident set holds (-1: empty).  In every
 * kvo_decode_step, per layer: (urgent) the true index T becomes resident --
 * blocks already resident stay in their slots, the missing ones in ascending
 * id order take the reusable slots in ascending slot order, a slot being
 * reusable when empty or holding a block neither in T nor in the prediction P
 * fetched for this step -- and only those blocks cross the host link, on the
 * urgent stream; attention reads T through its slots; then (prefetch, with a
 * speculative query) the prediction for the next step becomes resident the
 * same way, sparing the blocks of T, on the low-priority stream.  Without a
 * speculative query only the urgent phase runs (the previous step's T is
 * spared); when moreover no prefetch is in flight and no layer has low-rank
 * keys, the step is one chain on the compute stream, and kvo_set_graphs(1)
 * replays it from a CUDA graph.  In a chain step attention is split: the
 * blocks of T that were resident already, and the window, are attended while
 * the urgent copy runs (the TMA-staged kernel, launched as a programmatic
 * dependent of the copy so that it takes the SMs the copy leaves free), then
 * the fetched blocks, merged into the first result by log-sum-exp (with the
 * register-direct attention kernel, kvo_set_attn_impl 0, the step attends to
 * the whole set after the copy instead).  A step with a speculative query and
 * no low-rank layer splits its attention the same way, the first part
 * launched plainly on a stream of its own (compute priority) once the
 * blocks prefetched for the step have landed.  The copies of this mode always use
 * the flat gather engine (engine 3, with per-entry destination slots)
 * whatever kvo_set_gather_engine chose.
 *   kvo_resident_slots: synchronize, copy layer `layer`'s slot table
 *   [G][2k] int32 to host memory `slots_out`.
 *   kvo_resident_fetched: synchronize, write the blocks fetched since init (or
 *   the last reset) to host out2[0] (urgent) and out2[1] (prefetch); reset != 0
 *   zeroes the counters afterwards.
 *   Errors: KVO_ERR_STATE when the context was built with resident = 0;
 *   KVO_ERR_INVALID for a bad layer or a null pointer.
 */
/*
 * kvo_set_prefetch_budget -- admission cap on the host bytes of speculation
 * (resident = 1; PulseInfer §2 names I/O-adaptive offloading admission
 * without a rule): each prefetch phase fetches at most `blocks` missing blocks
 * per (request, KV head) and layer, those with the lowest ids; -1 (default)
 * admits all.  The urgent phase is never capped, so results do not change:
 * a block the cap left out that the true index needs is fetched urgently.
 * Synchronizes the context's streams.  Errors: KVO_ERR_STATE with
 * resident = 0; KVO_ERR_INVALID for blocks < -1.
 */
kvo_status kvo_set_prefetch_budget(kvo_ctx* ctx, int blocks);

/*
 * kvo_set_spec_policy -- when the speculative prefetch runs (resident = 1,
 * steps with a speculative query).  mode 0 (default): every layer prefetches
 * its prediction for the next step.  mode 1: per layer, only while it pays.
 * The resident assign kernel counts, per layer, the blocks its prefetch phase
 * fetched and those of them a later true index used; a used prefetch saves an
 * urgent fetch, an unused one costs a fetch, so prefetching lowers the host
 * bytes only while more than half of the prefetched blocks are used.  The
 * decision is taken on the GPU, in stream order, by the last CTA of each
 * layer's urgent assign: a layer whose prefetches were used less over a window
 * of 4 steps fetches nothing in its prefetch phase for the next 32 steps, then
 * tries again (the rest doubles after every try that fails, up to 1024 steps,
 * and returns to 32 after a window that pays).  Outputs never depend on the policy (a block the true index
 * needs is fetched urgently when missing).
 * Synchronizes the context's streams.  Errors: KVO_ERR_STATE with
 * resident = 0; KVO_ERR_INVALID for a mode outside 0..1.
 *
 * kvo_spec_stats -- synchronize, then write per layer l to host out3[3 l ..]:
 * blocks prefetched since init, prefetched blocks a true index used, and 1 if
 * the layer's prefetch phase is on (always 1 with mode 0).
 * Errors: KVO_ERR_STATE with resident = 0; KVO_ERR_INVALID for a null output.
 */
kvo_status kvo_set_spec_policy(kvo_ctx* ctx, int mode);
kvo_status kvo_spec_stats(kvo_ctx* ctx, int64_t* out3);

/*
 * kvo_set_lowrank_keys -- rebuild the keys of a layer's missed blocks on the
 * GPU instead of fetching them (DualDecoder §5.3: low-rank key reconstruction
 * from a GPU-resident low-rank key cache; only the values of missed blocks
 * then cross the host link).
 *   coef: device bf16, packed like the host K cache with rank entries per
 *     token row instead of d: [b][Hkv][cap_b][rank].
 *   basis: device bf16 [b][Hkv][rank][d].
 *   Both caller-owned; they must stay valid while set.  Key row t of a group
 *   is bf16( sum over j = 0 .. rank-1 ascending of coef[t][j] * basis[j][c] ),
 *   each product and each partial sum rounded to fp32 (no fused multiply-add),
 *   the total rounded to bf16 to nearest-even; keys that are exactly this
 *   product (synthetic low-rank keys) are rebuilt bit for bit, other keys are
 *   replaced by their rank-`rank` image.
 *   Applies to the urgent phase of kvo_decode_step / kvo_decode_step_dual
 *   (both buffer modes); prefetches still copy K and V.  rank 0 turns it off.
 *   With kvo_append, the coefficient rows of appended tokens (rows len_b ..
 *   len_b + max_append - 1) are the caller's to fill before their blocks can
 *   be selected.
 *   Synchronizes the context's streams and drops captured graphs.
 *   Errors: KVO_ERR_INVALID for a bad layer, rank outside 0..64, or null
 *   factors with rank > 0.
 */
kvo_status kvo_set_lowrank_keys(kvo_ctx* ctx, int layer, int rank, const void* coef, const void* basis);
kvo_status kvo_resident_slots(kvo_ctx* ctx, int layer, int32_t* slots_out);
kvo_status kvo_resident_fetched(kvo_ctx* ctx, int64_t* out2, int reset);
kvo_status kvo_info(kvo_ctx* ctx, int64_t* out4);

/*
 * sparse_decode_attn_static -- sparse_decode_attn without a context and
 * without allocating device memory.  The pages have no counterpart to this
 * call; it exists for callers that cannot call cudaMalloc: code whose device
 * memory all belongs to another allocator (a framework arena or a pool sized
 * once at start-up), and latency-critical callers that cannot afford the
 * implicit device synchronisation of cudaMalloc / cudaFree in a decode loop.
 *   Inputs (device): q [b][Hq][d] bf16; k_buf, v_buf [G][2k][B][d] bf16 (the
 *   layout of a ping-pong half); slot_of_true [G][k] int32; k_win, v_win
 *   [b][Hkv][W][d] bf16 (may be NULL when W == 0).  Outputs as in
 *   sparse_decode_attn (fuse_window_merge picks one fused part or two parts);
 *   status (device int32, optional) receives KVO_DEV_BAD_SLOT for a slot
 *   outside [0, 2k), which is then not read (slot 0 is read in its place);
 *   with status == NULL such errors are dropped -- nothing reports them.
 *   The call cannot check buffer sizes (it has no context): each buffer must
 *   hold at least the elements its shape above implies.
 *   Scratch: one static device array of 24 MiB, reserved on every GPU that
 *   loads the library until the process exits.  A call needs
 *   items * r * (d + 2) * 4 bytes plus small tables, items = G * (ceil(k*B/256)
 *   + ceil(W/256)); larger calls are rejected with KVO_ERR_INVALID and a message
 *   giving both sizes.  Every call shares the array and leaves its contents
 *   behind (the tickets it needs are cleared at the start of each call), so
 *   calls that overlap on the GPU race: order them on one stream.
 *   The first call on each device looks up the array's device address with
 *   that device current (cudaGetSymbolAddress) and caches it; make that first
 *   call before any stream capture.  No cudaMalloc, cudaFree or allocating
 *   library routine is called.
 */
kvo_status sparse_decode_attn_static(const void* q, const void* k_buf, const void* v_buf,
                                     const int32_t* slot_of_true, const void* k_win, const void* v_win,
                                     float* o, float* lse, int32_t* status, int batch, int n_q_heads,
                                     int n_kv_heads, int head_dim, int block_size, int top_k, int window,
                                     int fuse_window_merge, kvo_stream_t stream);

/*
 * kvo_set_gather_shape -- launch shape of the host -> HBM gather kernel:
 * ctas (0: the default, 2 per SM), threads per CTA (32..256, multiple of 32)
 * and 16-byte loads of K and of V in flight per lane (1, 2 or 4).  The gather
 * reads host memory in place; its in-flight loads queue behind the host link,
 * so a shape that just saturates the link leaves the SMs' memory pipelines to
 * the HBM-bound kernels running beside it.
 */
kvo_status kvo_set_gather_shape(kvo_ctx* ctx, int ctas, int threads, int unroll);

/*
 * kvo_set_gather_engine -- how the gather moves bytes.  engine 0: lane loads
 * (the kernel shaped by kvo_set_gather_shape).  engines 1 and 2: TMA bulk
 * copies, host -> shared memory -> HBM, driven by `drivers` warps (0: default
 * 32), each with 3 (engine 1) or 7 (engine 2) batches of up to 16 KiB in
 * flight; the SMs' load/store pipelines stay free for the HBM-bound kernels
 * running beside it.  Every TMA wait is bounded (2 s); on expiry the driver
 * sets KVO_DEV_TIMEOUT and stops.  engine 3: lane loads over the index list
 * itself, a flat stream of 16-byte words per group (entry j of a list goes to
 * slot base + j, so adjacent ids are read and written as contiguous ranges);
 * the decode step then skips building run lists.  Engine 3 is the default:
 * 38 CTAs x 1024 threads, 2 loads of K and of V in flight per lane, 200 KiB of
 * shared memory reserved per CTA so each gather CTA has an SM to itself.
 * engine 4: the copy engine -- the run list is read back to pinned host
 * memory (the call synchronizes its stream for it) and every run becomes one
 * cudaMemcpyAsync of K and one of V on the stream, issued by the host: no SM
 * moves a byte, but the host issues two calls per run and waits for the run
 * list inside each gather (so decode steps with engine 4 are never captured
 * into graphs; kvo_set_graphs(1) then fails with KVO_ERR_STATE).
 * Selecting an engine resets the launch shape to that engine's default.
 * Resident sets (resident = 1) always copy with engine 3.
 */
kvo_status kvo_set_gather_engine(kvo_ctx* ctx, int engine, int drivers);

/*
 * kvo_set_gather_reserve -- engine 3 only: shared memory each gather CTA
 * reserves without using it (0..232,320 bytes: 227 KiB less the kernel's own
 * 128-byte table).  A reservation near the SM's
 * capacity gives each gather CTA an SM of its own, so HBM-bound kernels never
 * share an SM (and its load/store pipeline) with loads waiting on the link.
 * Set the engine before kvo_set_gather_shape when asking for > 256 threads.
 */
kvo_status kvo_set_gather_reserve(kvo_ctx* ctx, int smem_bytes);

/*
 * kvo_set_attn_impl -- which kernel computes the attention of
 * sparse_decode_attn, sparse_decode_attn_cobatch and the decode step.  All
 * do the same arithmetic but split a group's tiles differently, so their
 * results agree up to float rounding, not bit for bit.
 * impl 0: register-direct, one CTA per 256-token work item, each warp loading
 * its tiles' K/V fragments from HBM with 16-byte loads.
 * impl 1: TMA-staged persistent kernel; each of a CTA's four warps keeps its
 * next 2-4 tiles in flight in shared-memory stages filled by bulk copies, and
 * the tiles of all groups are split into one equal contiguous range per CTA,
 * over as many CTAs as are resident on the device at once (in the decode step:
 * on the SMs the flat gather leaves free), or over `ctas` CTAs when ctas > 0.
 * impl 2 (default): group-split clusters for the fused output (the window
 * merged in; "Scaling Attention Beyond GPUs for LLM Inference", abstract): a
 * cluster of S CTAs per (request, KV head) group splits the group's tiles,
 * attends with one softmax over both parts and merges the CTAs' states through
 * distributed shared memory, with no partial results in global memory.
 * ctas = S (1..8), or 0: S = the resident CTA slots / groups (at most 8), and
 * clusters only where the groups' CTAs then fill at least 3/4 of the slots --
 * otherwise, and for separate parts (fuse_window_merge = 0), impl 1 runs.
 * Waits inside impls 1 and 2 are bounded (2 s); on expiry the kernel sets
 * KVO_DEV_TIMEOUT.  Synchronises the context's streams and drops captured
 * graphs.  Errors: KVO_ERR_INVALID for a null context, impl outside 0..2,
 * ctas < 0, or ctas > 8 with impl 2; KVO_ERR_CUDA if the work lists cannot be
 * allocated.
 */
kvo_status kvo_set_attn_impl(kvo_ctx* ctx, int impl, int ctas);

/*
 * kvo_set_select_impl -- which kernel computes select_topk and the decode
 * step's selection.  Both compute the exact top-k (DualDecoder §4.1, Fig. 6)
 * and give identical indices.  A group's landmark rows are split over CTAs of
 * 256 threads x 1, 2 or 4 rows (the same split for every group).
 * impl 0: the CTAs score their rows into global keys and histograms; the last
 * CTA of each group (an atomic ticket) selects on its own.
 * impl 2: where every group's CTAs number at most 8 they form one
 * thread-block cluster per group; each keeps its keys in shared memory and
 * the radix select runs on all of them, exchanging digit histograms and
 * winner counts through distributed shared memory (nothing through global
 * memory).  Otherwise impl 0 runs.
 * impl 1 (default): impl 2 where the ticket kernel's tail would be long and
 * exposed (groups of more than 1024 blocks and a grid that fits one wave of
 * 4 CTAs per SM), else impl 0.
 * Synchronises the context's streams and drops captured graphs.  Errors:
 * KVO_ERR_INVALID for a null context or impl outside 0..2.
 */
kvo_status kvo_set_select_impl(kvo_ctx* ctx, int impl);

/*
 * kvo_plan_select -- the selection kernels' launch plan for a shape, computed
 * on the host: no context, no GPU.  blocks_per_group[n_groups] (host int32,
 * >= 0): each group's candidate blocks at capacity (C_b, or the count it may
 * grow to).  n_sms: the device's SMs (each holds 4 selection CTAs of 256
 * threads).  impl: as kvo_set_select_impl.  Writes host out4 = {rows per
 * thread (1, 2 or 4: 1024 rows per CTA when that gives about 8 CTAs per SM
 * or more, else 512 or 256, whichever needs fewer waves, 256 on a tie), the
 * most CTAs a group needs, the CTAs of the ticket kernel's grid, the CTAs per
 * cluster of the cluster kernel or 0 when the ticket kernel runs}.
 * Errors: KVO_ERR_INVALID for n_groups or n_sms <= 0, impl outside 0..2, a
 * negative count or a null pointer.
 */
kvo_status kvo_plan_select(int n_groups, const int32_t* blocks_per_group, int n_sms, int impl, int32_t* out4);

/*
 * kvo_plan_attention -- the work split of the TMA-staged attention kernel
 * (kvo_set_attn_impl 1) for a shape, computed on the host: no context, no GPU.
 * The tiles (16 tokens) of every group -- its sparse part of sparse_tokens
 * (k * block_size), then its window part of window_tokens (W, or W + B - 1
 * when the cache grows) -- are laid out group after group and split into
 * `grid` contiguous ranges of equal cost (a tile costs 1, entering a part 12
 * more: the work-item epilogue), range bounds rounded down to a multiple of
 * the CTA's 4 warps; each range is cut at part boundaries into work items.
 *   n_groups: b * Hkv.  grid: CTAs asked for; the plan uses min(grid, tiles).
 *   items_out: host [items_cap][4] int32, nullable: {group, part (0 sparse,
 *     1 window), first tile within the part, tiles}, in range order.
 *   cta_out: host [grid + 1] int32, nullable: first item of each range, then
 *     the item count.
 *   n_items_out, grid_out: host, the item count and the grid used.
 * Call once with items_out = NULL to size the buffers.  Errors:
 * KVO_ERR_INVALID (message via kvo_last_error(NULL)) for n_groups or grid <= 0,
 * negative token counts, both zero, null count pointers, or items_cap below the
 * item count when items_out is given.
 */
kvo_status kvo_plan_attention(int n_groups, int sparse_tokens, int window_tokens, int grid, int32_t* items_out,
                              int items_cap, int32_t* cta_out, int32_t* n_items_out, int32_t* grid_out);

/*
 * Per-launch timing of kvo_decode_step, for benchmarks.  kvo_profile(ctx, 1)
 * clears and starts recording a timing event before and after every kernel
 * the step launches, on the stream it runs on; kvo_profile(ctx, 0) stops.
 * kvo_profile_read synchronizes, then writes per kernel kind the summed
 * launch durations (ms) and launch counts, and clears the record.  Kinds:
 * 0 select (with resident = 1 and no speculative query, the urgent residency
 * assignment runs inside it), 1 index diff (and residency assignment), 2 run coalescing,
 * 3 prefetch gather, 4 urgent gather, 5 attention, 6 low-rank key
 * reconstruction (n_kinds >= 7).
 */
kvo_status kvo_profile(kvo_ctx* ctx, int enable);
kvo_status kvo_profile_read(kvo_ctx* ctx, double* ms_out, int64_t* launches_out, int n_kinds);
/* kvo_profile_trace: the recorded launches in issue order (call before
 * kvo_profile_read, which clears them): start and end (ms, relative to the
 * first recorded launch), kind and layer.  Writes min(cap, count) entries and
 * the count to *n_out. */
kvo_status kvo_profile_trace(kvo_ctx* ctx, double* start_ms, double* end_ms, int32_t* kind, int32_t* layer,
                             int cap, int* n_out);

/*
 * kvo_set_wait_test -- for testing the bounded waits of the TMA-staged
 * attention kernel (kvo_set_attn_impl 1).  limit_ns (1 ms .. 10 s; default
 * 2 s) bounds every mbarrier wait of that kernel.  skip_tile >= 0 makes the
 * first warp of CTA 0 in every later launch announce its tile number skip_tile
 * (counted from 0 in that warp's own order) without copying it, so the wait
 * for that tile runs out: the kernel then sets KVO_DEV_TIMEOUT in the device
 * status word, stops waiting and issuing, lets every copy it did issue land,
 * and returns; its outputs are invalid.  skip_tile = -1 (default) copies everything.  Synchronizes the
 * context's streams and drops captured graphs.  Errors: KVO_ERR_INVALID for
 * limit_ns outside 1 ms .. 10 s or skip_tile < -1.  Not for production use.
 */
kvo_status kvo_set_wait_test(kvo_ctx* ctx, int64_t limit_ns, int skip_tile);

/* Human-readable description of the last error of ctx (or of the last
 * context-free call when ctx is NULL).  Never NULL. */
const char* kvo_last_error(const kvo_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* KVO_H */
