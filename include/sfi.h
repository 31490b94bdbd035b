/*
 * sfi.h -- C ABI of the Slow-Fast Inference (SFI) decode-attention path on sm_103a.
 *
 * The path (arXiv 2603.12038, "Slow-Fast Inference: Training-Free Inference Acceleration
 * via Within-Sentence Support Stability"; sections cited below are from the gist.science
 * technical summary of that paper unless named otherwise):
 *   every step   sfi_append_kv            write the new token's K/V row
 *   slow step    sfi_dense_decode_attn    dense attention + per-position evidence
 *                sfi_select               evidence + positional prior -> Top-K positions
 *                sfi_compact              pack sinks + selected rows contiguously
 *   fast step    sfi_sparse_decode_attn   attention over the packed rows + recent window
 *                sfi_fast_decode_step     the append and that attention in one launch
 *   host         sfi_schedule             trigger policy: slow or fast for each step
 *
 * Conventions for every call:
 *   - All tensors are device memory owned by the caller; the library never allocates.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *     default stream) and never synchronise, except sfi_read_error.
 *   - Argument errors are returned synchronously, before anything is launched.
 *   - A failed launch returns SFI_ERR_CUDA (from cudaGetLastError).
 *   - Kernels that find bad device-side data (a page-table entry out of range, an append
 *     past capacity, a bounded wait that gave up) set bits in the caller's device error
 *     word `err` and skip the bad access; they never trap. Read it with sfi_read_error.
 *   - The library keeps no state between calls except per-device tables (the resolved
 *     driver entry point, cluster occupancy), the scratch of
 *     sfi_sparse_decode_attn_static and the one-shot sfi_test_inject_stall flag; calls
 *     sharing one workspace must not overlap on the GPU.
 *   - Shapes: head_dim must be 128; group = n_q_heads / n_kv_heads must be 1, 2, 4 or 8;
 *     batch <= 256. Query head h belongs to kv head h / group. A "unit" is one
 *     (layer, sequence, kv head), numbered u = (layer * batch + b) * n_kv_heads + kv_head.
 *   - bf16 pointers must be 16-byte aligned.
 */
#ifndef SFI_H
#define SFI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sfi_status {
    SFI_OK = 0,
    SFI_ERR_INVALID_ARG = 1,  /* null pointer, inconsistent shape, misaligned pointer     */
    SFI_ERR_UNSUPPORTED = 2,  /* head_dim != 128, group not in {1,2,4,8}, batch > 256       */
    SFI_ERR_CAPACITY = 3,     /* a host-known length bound exceeds a buffer's capacity      */
    SFI_ERR_WORKSPACE = 4,    /* workspace missing, too small or not 256-byte aligned      */
    SFI_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed               */
    SFI_ERR_DEVICE = 6        /* sfi_read_error: the device error word is non-zero          */
} sfi_status;

/* Bits of the device error word. */
#define SFI_DEVERR_PAGE_RANGE 0x1u /* page-table entry outside [0, n_pages): access skipped  */
#define SFI_DEVERR_CAPACITY 0x2u   /* append at a position >= capacity: row not written      */
#define SFI_DEVERR_TIMEOUT 0x4u    /* a bounded pipeline wait gave up: outputs invalid,      */
                                   /* re-initialise the workspace before further use         */
#define SFI_DEVERR_LENGTH 0x8u     /* seq_len[b] > max_len: that sequence's work skipped     */

/*
 * The KV cache of all layers (summary section 3: recent tokens are read straight from the
 * paged KV cache). Two layouts:
 *   page_size == 0  contiguous  k, v: bf16 [n_layers][batch][n_kv_heads][capacity][128]
 *   page_size == 16 paged       k, v: bf16 [n_layers][n_pages][n_kv_heads][16][128];
 *                               position p of sequence b lives in page
 *                               page_table[b * max_pages_per_seq + p / 16], row p % 16;
 *                               capacity = max_pages_per_seq * 16.
 * seq_len (device int32 [batch]) holds each sequence's current length; sfi_append_kv writes
 * at seq_len[b] and increments it. max_len is a host-known upper bound of every seq_len
 * entry during the call (used only to size grids and check capacity). err is a device
 * uint32 error word, shared by every call that gets this descriptor.
 */
typedef struct sfi_kv_cache {
    int32_t n_layers, batch, n_q_heads, n_kv_heads, head_dim;
    int32_t capacity;
    int32_t page_size;
    int32_t n_pages;
    int32_t max_pages_per_seq;
    int32_t max_len;
    void *k;
    void *v;
    const int32_t *page_table;
    int32_t *seq_len;
    uint32_t *err;
} sfi_kv_cache;

/*
 * Sparse-state budget (summary 2A: sink tokens + sliding recent window + selected memory)
 * and Selector parameters (summary 2B: fused score s = (1 - lambda) f + lambda r).
 * prior_tau is the ramp length of the positional prior and must be a power of two.
 */
typedef struct sfi_budget {
    int32_t n_sink;
    int32_t n_window;
    int32_t n_select;
    int32_t prior_tau;
    double lambda;
    /* Selector refinements, read by sfi_refine_scores only (each is off when zero):     */
    int32_t nms_radius;  /* Soft-NMS: neighbours at distance 1..nms_radius in a head     */
    float nms_gamma;     /* Soft-NMS: factor for a candidate that a neighbour suppresses */
    float excl_mu;       /* cross-head exclusivity strength in [0, 1]                    */
    float norm_nu;       /* key-norm prior term: prior scaled by min(1, norm_nu/||k||)   */
    int32_t geometric;   /* 1: geometric (log-linear) mixture instead of arithmetic      */
    float nms_delta;     /* Soft-NMS: only a neighbour at most nms_delta above suppresses */
                         /* (scores that similar); 0 = any strictly higher neighbour     */
} sfi_budget;

/*
 * The packed sparse memory (summary section 3: sinks and selected tokens are packed into
 * one contiguous buffer after every slow step).
 *   kc, vc   bf16 [n_layers][batch][n_kv_heads][n_sink + n_select][128]
 *   sel_idx  int32 [n_layers][batch][n_kv_heads][n_select]  ascending positions (sfi_select)
 *   sel_cnt  int32 [n_layers][batch][n_kv_heads]            valid entries of sel_idx
 *   rows     int32 [n_layers][batch][n_kv_heads]            packed rows = sinks + sel_cnt
 *                                                           (written by sfi_compact)
 */
typedef struct sfi_sparse_mem {
    void *kc;
    void *vc;
    int32_t *sel_idx;
    int32_t *sel_cnt;
    int32_t *rows;
} sfi_sparse_mem;

/* Human-readable name of a status code (static storage). */
const char *sfi_status_string(sfi_status s);

/* Library version string (static storage). */
const char *sfi_version(void);

/*
 * Bytes of device workspace that sfi_dense_decode_attn and sfi_sparse_decode_attn need
 * for this cache shape on the current device: split-KV partials, per-unit tickets,
 * per-unit softmax statistics and the dense step's fp32 logits
 * ([units][capacity][group]). 0 on invalid arguments.
 */
size_t sfi_workspace_bytes(const sfi_kv_cache *kv, const sfi_budget *budget);

/* Zero a workspace (its tickets must start at zero). Call once after allocating it, and
 * again after a SFI_DEVERR_TIMEOUT. Asynchronous on stream. */
sfi_status sfi_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * Append one token per sequence (implied by every decode step; summary section 1).
 * k_new, v_new: bf16 [n_layers][batch][n_kv_heads][128]. For each sequence b with
 * active[b] != 0 (active: device uint8 [batch], NULL = all), writes row seq_len[b] of every
 * (layer, kv head) and then increments seq_len[b]. Requires max_len + 1 <= capacity.
 */
sfi_status sfi_append_kv(const sfi_kv_cache *kv, const void *k_new, const void *v_new,
                         const uint8_t *active, void *stream);

/*
 * Slow step: dense decode attention (blog, "How SFI Works": the slow step attends to the
 * whole KV cache; summary 2A "Slow Steps"). For every unit of an active sequence, each of
 * its `group` query heads h computes
 *     z_hj = q_h . k_j / sqrt(128),  p_hj = softmax_j(z_h),  o_h = sum_j p_hj v_j
 * over j in [0, seq_len[b]). Split-KV: persistent CTAs stream contiguous tile ranges and the
 * last CTA of a unit merges the partials.
 *   q        bf16 [n_layers][batch][n_q_heads][128]
 *   out      [n_layers][batch][n_q_heads][128], fp32 if out_fp32 else bf16
 *   scores_f optional fp32 [n_layers][batch][n_kv_heads][capacity]: the Selector's evidence
 *            (summary 2B "Evidenz") f_j = (1/group) sum_h p_hj for j < seq_len[b];
 *            NULL = dense-only, no emission.
 *   ws       workspace of at least sfi_workspace_bytes(), 256-byte aligned, initialised.
 */
sfi_status sfi_dense_decode_attn(const sfi_kv_cache *kv, const void *q, void *out,
                                 int32_t out_fp32, float *scores_f, const uint8_t *active,
                                 void *ws, size_t ws_bytes, void *stream);

/*
 * The Selector (summary 2B) for every unit of an active sequence of length L = seq_len[b]:
 * over the candidates j in [n_sink, L - n_window), with d_j = (L - n_window) - j and
 * n_C candidates,
 *     rt_j = fl32(min(1, d_j / prior_tau)),  Z = sum_j min(1, d_j / prior_tau)  (closed form)
 *     s_j  = fl32(fl32(c1 * f_j) + fl32(c2 * rt_j)),  c1 = fl32(1 - lambda), c2 = fl32(lambda/Z)
 * and keeps the min(n_select, n_C) largest s_j (ties to the lower position), written in
 * ascending position order to sel_idx with their count in sel_cnt. Radix select, one CTA
 * per unit. The sinks and the window are part of the sparse state by construction.
 */
sfi_status sfi_select(const sfi_kv_cache *kv, const float *scores_f, const sfi_budget *budget,
                      const sfi_sparse_mem *mem, const uint8_t *active, void *stream);

/*
 * Key norms for the Selector's key-norm prior term (summary 2B: the prior counters tokens
 * with extremely high key norms). norms: fp32 [n_layers][batch][n_kv_heads][capacity];
 * norms[u][j] = ||k_j||_2 for j < seq_len[b] of active sequences: squares of the bf16
 * values summed in fp32 in dimension order, then the correctly rounded square root.
 */
sfi_status sfi_key_norms(const sfi_kv_cache *kv, float *norms, const uint8_t *active,
                         void *stream);

/*
 * Refined Selector scores (summary 2B: the fused scores are refined by Soft-NMS within a
 * head and a soft cross-head competition before Top-K; the pages give no formulas, these
 * are the library's readings). For every (layer, sequence) of an active sequence and every
 * candidate j in [n_sink, L - n_window), all kv heads h:
 *   rt_hj = fl32(min(1, d_j / prior_tau)), times min(1, fl32(norm_nu / key_norms[h][j]))
 *           when norm_nu > 0 (key_norms may then not be NULL);
 *   s_hj  = arithmetic: fl32(fl32(c1 f_hj) + fl32(c2 rt_hj))  (c1, c2 as in sfi_select), or
 *           geometric:  fl32(c1 log2 f_hj) + fl32(lambda log2 fl32(fl32(c2 rt_hj) / lambda))
 *           in fp32 with the library's own log2 (log-domain score of the geometric mixture);
 *   Soft-NMS (a candidate is damped by a nearby one that scores a little higher): s'_hj =
 *           fl32(nms_gamma s_hj) if some candidate i with 1 <= |i - j| <= nms_radius has
 *           s_hi > s_hj and, when nms_delta > 0, fl32(s_hi - s_hj) <= nms_delta; else s_hj;
 *   exclusivity: s''_hj = fl32(s'_hj - fl32(mu' fl32(T_j - s'_hj))), T_j = sum over heads of
 *           s'_hj in head order, mu' = fl32(excl_mu / (n_kv_heads - 1)).
 * refined: fp32 [units][capacity], written at the candidate positions. Select on it with
 * sfi_select and lambda = 0 (which keeps the scores as they are). n_kv_heads <= 16, else
 * SFI_ERR_UNSUPPORTED. A negative nms_radius, nms_gamma or excl_mu outside [0, 1], a
 * negative or NaN nms_delta or norm_nu, or norm_nu > 0 without key_norms: SFI_ERR_INVALID_ARG.
 */
sfi_status sfi_refine_scores(const sfi_kv_cache *kv, const float *scores_f,
                             const float *key_norms, const sfi_budget *budget, float *refined,
                             const uint8_t *active, void *stream);

/*
 * Pack the sparse memory (summary section 3, memory-coalesced sparse kernel): for every
 * unit of an active sequence, copies the rows of the sinks [0, min(n_sink, L)) followed by
 * the selected positions sel_idx[0 .. sel_cnt) from the cache into kc/vc, and writes the
 * packed row count to mem->rows.
 */
sfi_status sfi_compact(const sfi_kv_cache *kv, const sfi_budget *budget,
                       const sfi_sparse_mem *mem, const uint8_t *active, void *stream);

/*
 * Inputs a fast step reads early. The fast-step calls (sfi_sparse_decode_attn,
 * sfi_fast_decode_step, sfi_sparse_decode_attn_static) start loading the packed memory (kc,
 * vc, rows, sel_cnt) and read `active` before they wait for the kernel issued before them on
 * the stream to finish (programmatic dependent launch). These must therefore be complete
 * when the call is issued. A kernel that writes them must not let its dependents start
 * before its writes: without programmatic dependent launch that is always so, and the
 * library's own sfi_select and sfi_compact let their dependents start only after their
 * writes. The query, the lengths and the new rows are read only after that wait.
 *
 * Fast step (blog, "How SFI Works": attention restricted to the support of the last slow
 * step; summary 2A "Fast Steps"): attention of each query head over the packed rows
 * kc/vc[0 .. mem->rows) of its unit plus the recent window [max(n_s, L - n_window), L) read
 * from the cache, where n_s = mem->rows - sel_cnt (the packed sinks) and L = seq_len[b].
 * Same q/out layouts and workspace as sfi_dense_decode_attn; no evidence is emitted.
 */
sfi_status sfi_sparse_decode_attn(const sfi_kv_cache *kv, const sfi_sparse_mem *mem,
                                  const sfi_budget *budget, const void *q, void *out,
                                  int32_t out_fp32, const uint8_t *active, void *ws,
                                  size_t ws_bytes, void *stream);

/*
 * A whole fast decode step in one launch (blog, "How SFI Works"; summary 2A "Fast Steps" and
 * section 3): the result of sfi_append_kv(kv, k_new, v_new, active) followed by
 * sfi_sparse_decode_attn(kv, mem, budget, q, out, ...). Each active sequence's new K and V
 * rows (k_new/v_new: device bf16 [n_layers][batch][n_kv_heads][128]) are written at position
 * seq_len[b] of the cache and attended as the last row of the recent window, and seq_len[b]
 * is advanced by one. kv->max_len bounds seq_len before the append (as for sfi_append_kv);
 * SFI_ERR_CAPACITY when max_len + 1 > capacity. Same q/out layouts, workspace and errors as
 * sfi_sparse_decode_attn. The workspace must have been cleared by sfi_workspace_init once;
 * calls leave its counters at zero again.
 */
sfi_status sfi_fast_decode_step(const sfi_kv_cache *kv, const sfi_sparse_mem *mem,
                                const sfi_budget *budget, const void *k_new, const void *v_new,
                                const void *q, void *out, int32_t out_fp32, const uint8_t *active,
                                void *ws, size_t ws_bytes, void *stream);

/*
 * The fast step for callers that cannot allocate device memory. The paper has no
 * counterpart of this call: it is an interface convenience. Some callers get only their
 * input and output buffers (for example a plug-in inside a host framework that owns all
 * device memory), or run a decode loop that must never call cudaMalloc because it may
 * synchronise the device; they cannot provide the workspace that sfi_sparse_decode_attn
 * needs.
 *
 * Same computation, arguments and layouts as sfi_sparse_decode_attn, minus the workspace.
 * The split-KV scratch (partials and per-unit tickets, about 2.1 MiB) lives in a fixed-size
 * device array inside the library, held by every GPU that loads the library until the
 * process exits. Limits: at most 16384 units (n_layers * batch * n_kv_heads), otherwise
 * SFI_ERR_CAPACITY and nothing is launched; at most 256 CTAs are used. The call allocates
 * nothing and calls no allocating routine; it clears the tickets it uses with an
 * asynchronous memset on `stream`.
 *
 * The first call on a device looks up the array's device address (once per device, with
 * that device current); make that first call before any stream capture. All calls share
 * the one array: calls whose execution overlaps on the GPU (different streams, or
 * different host threads without ordering) race and give wrong results.
 */
sfi_status sfi_sparse_decode_attn_static(const sfi_kv_cache *kv, const sfi_sparse_mem *mem,
                                         const sfi_budget *budget, const void *q, void *out,
                                         int32_t out_fp32, const uint8_t *active, void *stream);

/*
 * Trigger policy (summary 2C), host only: slow[t] = 1 when t == 0, when mask[t - 1] != 0
 * (the previous token is a boundary token), or when t_max > 0 steps have passed since the
 * last slow step. mask, slow: host uint8 [steps].
 */
sfi_status sfi_schedule(int32_t steps, const uint8_t *mask, int32_t t_max, uint8_t *slow);

/*
 * Trigger policy on the generated tokens (summary 2C: a slow step follows a trigger token
 * such as '.', '?', '!' or a newline), host only: slow[t] = 1 when t == 0, when
 * tokens[t - 1] is one of the n_trigger ids in trigger_ids, or when t_max > 0 steps have
 * passed since the last slow step. tokens: host int32 [steps]; slow: host uint8 [steps].
 */
sfi_status sfi_schedule_tokens(int32_t steps, const int32_t *tokens, const int32_t *trigger_ids,
                               int32_t n_trigger, int32_t t_max, uint8_t *slow);

/*
 * A whole decode run on one stream (blog "How SFI Works": the two-speed loop). For each
 * step t, with row t of k_new/v_new: for the sequences whose slow flag is set,
 * sfi_append_kv -> sfi_dense_decode_attn (with evidence) -> sfi_select -> sfi_compact, where
 * the append runs inside the dense launch (and, with a clustered Selector, the evidence is
 * computed by the Selector); for the others
 * sfi_fast_decode_step (append and sparse attention in one launch). Nothing is synchronised,
 * so the run can be captured in a CUDA graph and replayed (the caller restores seq_len before
 * each replay).
 *   slow      host uint8 [n_steps][batch], e.g. from sfi_schedule per sequence
 *   q         device bf16 [n_steps][n_layers][batch][n_q_heads][128]
 *   k_new/v_new device bf16 [n_steps][n_layers][batch][n_kv_heads][128]
 *   out       device [n_steps or 1][n_layers][batch][n_q_heads][128] (fp32 if out_fp32)
 *   scores_f  device fp32 [n_layers][batch][n_kv_heads][capacity] (evidence scratch)
 *   masks     device uint8 [n_steps][2][batch]: per-step (slow, fast) sequence masks, used
 *             when some step mixes slow and fast sequences; NULL if no step does
 *   len_start host bound of every seq_len before the first append
 *   dense_only 1: every step is append + dense attention without evidence (the full-KV
 *             baseline the pages compare against; the append fused into the dense
 *             launch); slow is ignored
 *   events    optional host array of 2 * n_steps cudaEvent_t (as void*): events[2t] and
 *             events[2t+1] are recorded (external, so they survive graph capture) right
 *             before and after step t's attention kernel (the fused fast step's kernel on
 *             fast steps, the dense kernel on slow ones; the whole slow step, joins
 *             included, with the layer-wise pipeline);
 *             NULL = none, and NULL entries are skipped
 *   side_stream layer-wise asynchronous pipeline (technical summary section 3, layer-wise
 *             overlap): NULL = off. When set, a slow step runs group of layers by group: dense
 *             attention and evidence of group i on `stream`, then sfi_select and sfi_compact
 *             of group i on side_stream, so that they overlap the attention of group i + 1;
 *             `stream` waits for side_stream before the step's last operation returns, so
 *             the next step sees the whole packed memory. A caller-owned stream of the same
 *             device; ignored when dense_only is set.
 *   fork_event, join_event  caller-owned cudaEvent_t (as void*, timing may be disabled),
 *             required with side_stream: fork_event is re-recorded on `stream` after each
 *             group's evidence and waited for on side_stream; join_event is recorded on
 *             side_stream after the last group and waited for on `stream`. Both work under
 *             stream capture (the usual fork/join of a captured graph). Missing events with
 *             side_stream set: SFI_ERR_INVALID_ARG.
 *   pipeline_group layers per dense launch with side_stream set (the Selector and packing of
 *             one group overlap the attention of the next): 0 = about a quarter of the layers
 *   concurrent_fast 1: on a step that mixes slow and fast sequences, the fast sequences'
 *             sfi_fast_decode_step runs on side_stream beside the slow sequences' Selector
 *             and packing on `stream`, forked after their dense launch (and evidence
 *             pass, if separate) (they touch disjoint sequences, packed memory and workspace
 *             regions); `stream` waits for side_stream before the step ends. Requires
 *             side_stream, fork_event and join_event (re-used per step as a fork and a
 *             join); replaces the layer-wise pipeline; 0 = off.
 *             events[2t], events[2t+1] then bracket the slow chain's dense kernel alone.
 * Results with the layer-wise pipeline equal those without up to the rounding of the dense
 * step's split-KV partition (one launch per group of layers instead of one for all layers);
 * with concurrent_fast they are bit-identical to the sequential run.
 */
typedef struct sfi_decode_plan {
    int32_t n_steps;
    const uint8_t *slow;
    const void *q;
    const void *k_new;
    const void *v_new;
    void *out;
    int32_t out_fp32;
    int32_t out_per_step;
    float *scores_f;
    const uint8_t *masks;
    int32_t len_start;
    int32_t dense_only;
    void *const *events;
    void *side_stream;
    void *fork_event;
    void *join_event;
    int32_t pipeline_group;
    int32_t concurrent_fast;
} sfi_decode_plan;

sfi_status sfi_decode_run(const sfi_kv_cache *kv, const sfi_budget *budget,
                          const sfi_sparse_mem *mem, const sfi_decode_plan *plan, void *ws,
                          size_t ws_bytes, void *stream);

/* Copy the device error word to *bits (synchronises `stream`). Returns SFI_OK when it is
 * zero, SFI_ERR_DEVICE when any bit is set. */
sfi_status sfi_read_error(const sfi_kv_cache *kv, uint32_t *bits, void *stream);

/* Clear the device error word (asynchronous). */
sfi_status sfi_clear_error(const sfi_kv_cache *kv, void *stream);

/*
 * Test hook for the bounded waits (no counterpart in the paper). With on != 0, the next
 * attention launch (sfi_dense_decode_attn, sfi_sparse_decode_attn, sfi_fast_decode_step or
 * one inside sfi_decode_run) makes its first CTA expect 16 bytes more on its first tile's
 * barrier than the copies deliver, so that barrier never completes: the waits on it give up
 * after about a second, SFI_DEVERR_TIMEOUT is set in the error word, the kernel drains its
 * copies and MMAs, frees its tensor memory and returns, and the context stays usable
 * (re-initialise the workspace before further use, as after any timeout). One-shot; process
 * wide. Not for production use.
 */
sfi_status sfi_test_inject_stall(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* SFI_H */
