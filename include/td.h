/*
 * td.h -- C ABI of the GB300 (sm_103a) decode-step library for TidalDecode's
 * Position Persistent Sparse Attention (PPSA).
 *
 * The method (TidalDecode: Fast and Accurate LLM Decoding with Position
 * Persistent Sparse Attention -- paper review page):
 *   - §三 "Position Persistent Sparse Attention": A = q K^T / sqrt(d),
 *     H = softmax(A) V per layer and head; sparse layers reuse the token
 *     positions chosen by the most recent selection layer instead of
 *     selecting per layer and head.
 *   - §二 "core insight" and §三 Figure 2: each decode step runs full
 *     attention at the first layers, full attention + top-k token selection
 *     at layer 2 and at one middle layer, and PPSA (sparse attention over the
 *     persisted positions) everywhere else.
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller; the
 *     library never allocates device memory on these paths.  Scratch comes
 *     from a caller-owned workspace of td_workspace_size() bytes that was
 *     zeroed once by td_workspace_init() (kernels leave it re-usable).
 *   - Layouts (row-major, contiguous):
 *       q          [batch][num_q_heads][head_dim]                 bf16
 *       k/v cache  [batch][num_kv_heads][max_seq_len][head_dim]   bf16
 *       seq_lens   [batch]                                        int32 (device)
 *       out        [batch][num_q_heads][head_dim]                 bf16
 *       out_f32    [batch][num_q_heads][head_dim]                 fp32 (optional)
 *       idx        [batch][num_kv_heads][top_k]                   int32
 *       scores     [batch][num_kv_heads][max_seq_len]             fp32 (optional)
 *     Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *     q, k, v, out and out_f32 must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = legacy default stream).  Outputs are valid once the stream has
 *     reached the end of the call.  Calls that share a workspace must be
 *     ordered on one stream.
 *   - Errors: argument, shape and schedule errors are detected on the host
 *     before anything is launched and returned synchronously.  A failed
 *     launch returns TD_ERR_CUDA.  Device-side input errors (an index at or
 *     beyond seq_lens[b], a seq_lens entry outside [0, max_seq_len]) never
 *     fault: the offending entry is skipped or clamped and a bit is set in
 *     the workspace status word, read with td_workspace_status().
 *   - No C++ exception crosses this interface.
 */
#ifndef TD_H_
#define TD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TD_OK = 0,
    TD_ERR_INVALID_ARG = 1,         /* null/misaligned pointer, bad count or mode */
    TD_ERR_UNSUPPORTED_SHAPE = 2,   /* head_dim != 128, group size not 1/2/4/8, ... */
    TD_ERR_NO_SELECTION = 3,        /* sparse layer with no persisted index set */
    TD_ERR_WORKSPACE_TOO_SMALL = 4,
    TD_ERR_CUDA = 5                 /* a CUDA runtime call or launch failed */
} td_status;

/* Layer modes of one decode step (review §三 Figure 2). */
typedef enum {
    TD_MODE_FULL = 0,          /* full attention, no selection            */
    TD_MODE_FULL_SELECT = 1,   /* full attention + top-k token selection  */
    TD_MODE_SPARSE = 2         /* PPSA: attention over the persisted set  */
} td_layer_mode;

/* Bits of the device status word (td_workspace_status). */
#define TD_FLAG_INDEX_OUT_OF_RANGE 0x1u   /* idx entry < -1 or >= seq_lens[b]: skipped */
#define TD_FLAG_SEQ_LEN_OUT_OF_RANGE 0x2u /* seq_lens[b] < 0 or > max_seq_len: clamped */
#define TD_FLAG_WAIT_TIMEOUT 0x4u         /* a staged kernel's bounded wait for its copies gave up;
                                             that (batch, KV head)'s output lacks the tokens of
                                             the CTA that gave up (the workspace stays usable) */

typedef struct {
    int32_t batch;          /* B  >= 1                                         */
    int32_t num_q_heads;    /* Hq >= 1, a multiple of num_kv_heads             */
    int32_t num_kv_heads;   /* Hkv >= 1; Hq / Hkv must be 1, 2, 4 or 8         */
    int32_t head_dim;       /* d; only 128 is supported                        */
    int32_t max_seq_len;    /* N_max: token rows per (batch, KV head) in K/V   */
    float scale;            /* softmax scale; 0 selects 1/sqrtf(head_dim)      */
} td_shape;

/* Human-readable name of a status code (static storage). */
const char *td_status_string(td_status status);

/* Bytes of workspace needed by every call below for this shape and top_k
 * (top_k = 0 when no call selects or runs sparse attention).  Returns 0 for
 * an invalid shape.  Does not touch the GPU. */
size_t td_workspace_size(const td_shape *shape, int32_t top_k);

/* Zero a freshly allocated workspace (a cudaMemsetAsync on `stream`).  Must
 * be called once before the workspace's first use; the kernels leave it
 * in the same state after every call. */
td_status td_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Synchronise `stream`, copy the device status word into *flags
 * (TD_FLAG_* bits, 0 = clean) and clear it. */
td_status td_workspace_status(void *ws, size_t ws_bytes, uint32_t *flags, void *stream);

/*
 * One full-attention layer, optionally with token selection (review §三
 * Figure 2 rows "Full Attention" and "Full Attention + Token Selection").
 *   For every batch row b and query head h, with a[n] = scale * q[b,h] . K[b,g(h),n]
 *   for n < seq_lens[b]:   out[b,h] = sum_n softmax(a)[n] * V[b,g(h),n].
 *   top_k > 0 also selects, per (b, KV head g), the top_k positions by the
 *   summed score s[n] = sum over the query heads h of g of a_h[n]; ties go
 *   to the lower position; idx_out[b,g,:] receives them in ascending order,
 *   padded with -1 when seq_lens[b] < top_k.
 *   top_k = 0: no selection (idx_out may be NULL).
 *   out_f32 (optional) receives the fp32 result before rounding to bf16.
 *   scores_out (optional, fp32 [B][Hkv][max_seq_len]) receives s[n] for
 *   n < seq_lens[b] when top_k > 0 (other entries untouched).
 *   A batch row with seq_lens[b] = 0 gets out = 0.
 */
td_status td_full_attn_select(const td_shape *shape, const void *q, const void *k_cache,
                              const void *v_cache, const int32_t *seq_lens, int32_t top_k,
                              int32_t *idx_out, void *out, float *out_f32, float *scores_out,
                              void *ws, size_t ws_bytes, void *stream);

/*
 * The selection step of a FULL_SELECT layer on its own, from caller-provided
 * scores (review §二 core insight: keep the tokens with the highest
 * attention scores; §三 Figure 2 "Token Selection -> top-k tokens").
 *   scores   device fp32 [B][Hkv][max_seq_len]; entries n < seq_lens[b] are read.
 *   idx_out  device int32 [B][Hkv][top_k]: per (b, g) the top_k positions of
 *            the largest scores, ties to the lower position, ascending,
 *            padded with -1 when seq_lens[b] < top_k.  -0.0 ties with +0.0;
 *            NaN scores give an unspecified (but in-range) selection.
 *   top_k >= 1.  The workspace is used for its status word only.
 */
td_status td_topk_select(const td_shape *shape, const float *scores, const int32_t *seq_lens,
                         int32_t top_k, int32_t *idx_out, void *ws, size_t ws_bytes,
                         void *stream);

/*
 * A selection layer with a coverage budget instead of a fixed k ("Dynamic
 * Token Coverage", Token Sparse Attention §2: rank the tokens by importance
 * and prune the least important while the pruned attention mass stays within
 * tau).  Full attention as td_full_attn_select; then per (batch row, KV
 * head), with s the selection scores over the row's N_b positions:
 *   k = min(k_max, the smallest k whose k highest scores hold at least 1 - tau
 *       of softmax(s)),
 * and the k positions with the highest scores (ties to the lower position)
 * are written ascending to idx_out[b][g][0..k), the rest of the row -1.
 *   tau in [0, 1); k_max >= 1 is the row length of idx_out [B][Hkv][k_max]
 *   (size the workspace with td_workspace_size(shape, k_max)).
 *   counts_out: device int32 [B][Hkv] (optional): k per row.
 * The mass sums are fp32: where the cumulative mass at the cut is within
 * rounding of 1 - tau, k may differ by one from an exact computation.  For
 * grouped-query heads s is the summed logit of the group (as for top-k), so
 * the mass is that of softmax over the summed logits.
 */
td_status td_full_attn_select_coverage(const td_shape *shape, const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *seq_lens, float tau,
                                       int32_t k_max, int32_t *idx_out, int32_t *counts_out,
                                       void *out, float *out_f32, float *scores_out, void *ws,
                                       size_t ws_bytes, void *stream);

/*
 * Overlap of two index sets, per (batch row, KV head): counts[b][g] =
 * |A[b][g] ∩ B[b][g]|, the number of positions present in both.  This is the
 * measure behind the review's token-selection sensitivity analysis (§三
 * "Token selection layer sensitivity", Figure 4(a): the overlap of the most
 * attended tokens between consecutive layers); the overlap rate is
 * counts / |A|, with |A| the number of entries >= 0 (min(top_k, N_b) for a
 * set the library wrote).
 *   idx_a, idx_b: device int32 [B][Hkv][top_k], each row ascending with -1
 *     padding only at its end (the layout td_full_attn_select writes);
 *     entries are positions, compared by value.
 *   counts: device int32 [B][Hkv] (written, caller-owned).
 *   top_k >= 1.  Shape as for the other calls (seq_lens are not needed).
 * Asynchronous on `stream`.  Errors: TD_ERR_INVALID_ARG for null or
 * misaligned pointers or top_k < 1; TD_ERR_CUDA if the launch fails.  A row
 * that is not ascending gives an unspecified count (no fault).
 */
td_status td_index_overlap(const td_shape *shape, const int32_t *idx_a, const int32_t *idx_b,
                           int32_t top_k, int32_t *counts, void *stream);

/*
 * One PPSA layer (review §三 "Position Persistent Sparse Attention"):
 *   attention of every query head over the positions idx[b,g(h),0..top_k)
 *   only (entries of -1 are padding and are skipped), with the softmax
 *   normalised over those positions.  An all-padding row gives out = 0.
 *   idx entries must be distinct; their order does not matter.
 */
td_status td_sparse_attn(const td_shape *shape, const void *q, const void *k_cache,
                         const void *v_cache, const int32_t *seq_lens, const int32_t *idx,
                         int32_t top_k, void *out, float *out_f32, void *ws, size_t ws_bytes,
                         void *stream);

/*
 * td_sparse_attn for callers that cannot allocate device memory.  The paper
 * has no counterpart: this is a deployment variant of the PPSA layer above,
 * with the same arguments minus the workspace.  It runs the kernel
 * td_sparse_attn runs by default (tensor cores for G = 4, 8; CUDA cores
 * otherwise) with a split plan of its own (about 256 index entries per CTA,
 * fewer splits when the scratch would not hold their partials), so its
 * result agrees with td_sparse_attn's within the parity tolerance (bf16
 * max-abs 2e-2, fp32 row-relative 1e-5), not bit for bit.
 *
 * Who needs it: code that may not call cudaMalloc or own a workspace -- a
 * component inside a host framework that hands out all device memory from
 * its own arena, a latency-critical path that must never enter the driver's
 * allocator (it can synchronise the device), a plugin whose memory budget is
 * fixed before it is loaded.  The entry point allocates nothing: its scratch
 * (split partials, arrival tickets, status word) is one fixed array of
 * TD_NOALLOC_SCRATCH_BYTES bytes inside the library's device image, which
 * every GPU that loads the library keeps until the process exits.
 *   - The first call on a device looks up the array's address (per device,
 *     with that device current) and caches it for the CUDA context current
 *     then; a later call in another context (after cudaDeviceReset, say)
 *     looks it up again.  Make the first call in each context before any
 *     stream capture starts.
 *   - Every call shares the array, which keeps the last call's contents; each
 *     call clears the parts that must start at zero on its own stream.  Calls
 *     whose kernels overlap on the GPU race on the array: keep them ordered on
 *     one stream.
 *   - Shapes whose scratch would exceed the array return
 *     TD_ERR_WORKSPACE_TOO_SMALL before anything is launched.  A shape whose
 *     top_k fits one CTA (at most 2048 entries) needs only the tickets and the
 *     status word (4 bytes per (batch row, KV head)); more splits add
 *     (2 + 128) * 4 bytes per split and query head.
 *   - Out-of-range index entries are skipped as in td_sparse_attn; this entry
 *     point does not report the status word.
 */
#define TD_NOALLOC_SCRATCH_BYTES (8u << 20)
td_status td_sparse_attn_noalloc(const td_shape *shape, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *seq_lens,
                                 const int32_t *idx, int32_t top_k, void *out, float *out_f32,
                                 void *stream);

/*
 * One decode step over an L-layer attention-only stack (review §三 Figure 2).
 *   modes       HOST array [num_layers] of td_layer_mode.
 *   q, k_caches, v_caches, outs   HOST arrays of num_layers device pointers
 *               (one layer's tensors each, layouts as above).
 *   outs_f32    HOST array of num_layers device pointers (entries may be
 *               NULL), or NULL.
 *   idx_buf     device [B][Hkv][top_k]: the persisted index set.  Every
 *               FULL_SELECT layer overwrites it; every SPARSE layer reads the
 *               set of the most recent FULL_SELECT before it.  It stays on
 *               the device across layers and after the call.
 *   idx_valid   nonzero if idx_buf already holds a set on entry; otherwise a
 *               SPARSE layer before the first FULL_SELECT is rejected with
 *               TD_ERR_NO_SELECTION (nothing is launched).
 *   layer_events  optional HOST array of num_layers + 1 cudaEvent_t (as
 *               void*): event l is recorded on `stream` before layer l and
 *               event num_layers after the last layer (per-layer timing).
 * No host synchronisation happens inside the call; it can be captured into a
 * CUDA graph (see td_plan_create).
 */
td_status td_decode_step(const td_shape *shape, int32_t num_layers, const int32_t *modes,
                         const void *const *q, const void *const *k_caches,
                         const void *const *v_caches, const int32_t *seq_lens, int32_t top_k,
                         int32_t *idx_buf, int32_t idx_valid, void *const *outs,
                         float *const *outs_f32, void *ws, size_t ws_bytes, void *stream,
                         void *const *layer_events);

/*
 * A decode step captured once into a CUDA graph and replayed with one launch
 * (same arguments and semantics as td_decode_step; the pointers are baked
 * into the graph, so the buffers must stay allocated while the plan lives).
 * Creation runs no kernel.  td_plan_launch enqueues the whole step on
 * `stream`.  The plan holds host-side graph objects only.
 */
typedef struct td_plan td_plan;
td_status td_plan_create(td_plan **plan, const td_shape *shape, int32_t num_layers,
                         const int32_t *modes, const void *const *q,
                         const void *const *k_caches, const void *const *v_caches,
                         const int32_t *seq_lens, int32_t top_k, int32_t *idx_buf,
                         int32_t idx_valid, void *const *outs, float *const *outs_f32, void *ws,
                         size_t ws_bytes);
td_status td_plan_launch(td_plan *plan, void *stream);
void td_plan_destroy(td_plan *plan);

/*
 * td_plan_create_host: td_plan_create whose step also moves its inputs and
 * results between host and device, for callers whose q rows are produced,
 * and whose outputs are consumed, on the host.  The pages describe no such
 * call; it is the plumbing around the step.  Every layer's q rows and
 * outputs live in one buffer per side:
 *   q_host    HOST, page-locked (cudaHostAlloc / cudaHostRegister), bf16
 *             [num_layers][B][Hq][128]: copied to q at the start of the step.
 *   q         DEVICE bf16 [num_layers][B][Hq][128]: layer l reads q + l*B*Hq*128.
 *   outs      DEVICE bf16 [num_layers][B][Hq][128]: layer l writes outs + l*B*Hq*128.
 *   out_host  HOST, page-locked, bf16 [num_layers][B][Hq][128]: receives outs.
 * When both host buffers are mapped into the device's address space (as
 * page-locked memory is under unified addressing) and every buffer is
 * 16-byte aligned, kernels of the step copy over the chip-to-chip link in
 * its launch chain: q before layer 0 (beyond 1 MiB only layer 0's rows, the
 * rest by the copy engines on a second stream of the graph beside layer 0),
 * the outputs of every 8 layers by the copy engines on the second stream as
 * the step goes, the last two layers' by a kernel after the last layer.
 * Otherwise (or with the tuning key "host_copy" = 0 at creation) the copy
 * engines move them all: q in one copy before layer 0, the outputs of layers
 * 0 .. L-2 on the second stream while the last layer runs, the last layer's
 * after it.
 * Other arguments as in td_plan_create (outs_f32 stay on the device).
 * Pageable host memory is rejected with TD_ERR_INVALID_ARG (nothing
 * captured).  Each host range must lie in one page-locked allocation.  The
 * buffers must stay allocated while the plan lives; the step's results are
 * in out_host once the launch's stream has completed.
 */
td_status td_plan_create_host(td_plan **plan, const td_shape *shape, int32_t num_layers,
                              const int32_t *modes, const void *q_host, void *q,
                              const void *const *k_caches, const void *const *v_caches,
                              const int32_t *seq_lens, int32_t top_k, int32_t *idx_buf,
                              int32_t idx_valid, void *outs, float *const *outs_f32,
                              void *out_host, void *ws, size_t ws_bytes);

/*
 * KV append: the decode step's new token joins each layer's cache before
 * that layer attends (the growing KV cache of the decode phase, review §二).
 * seq_lens[b] already counts the new token, which sits at position
 * p_b = seq_lens[b] - 1.
 *   k_new, v_new   device bf16 [B][Hkv][128]: the new token's K and V rows
 *                  (16-byte aligned).
 *
 * td_kv_append writes k_new/v_new into k_cache/v_cache at p_b (rows with
 * seq_lens[b] outside [1, max_seq_len] are left alone).
 *
 * td_decode_step_append / td_plan_create_append: td_decode_step /
 * td_plan_create plus, per layer l, k_new[l] / v_new[l] (HOST arrays of
 * num_layers device pointers, both NULL for no append).  The step first
 * writes every layer's new rows (one launch per 32 layers), then attends:
 * full layers include position p_b, a sparse layer when p_b is in the
 * persisted set.  The result equals td_kv_append on every layer followed by
 * td_decode_step.  k_new/v_new may be written by the kernel just before the
 * call.
 */
td_status td_kv_append(const td_shape *shape, void *k_cache, void *v_cache, const void *k_new,
                       const void *v_new, const int32_t *seq_lens, void *stream);
td_status td_decode_step_append(const td_shape *shape, int32_t num_layers, const int32_t *modes,
                                const void *const *q, const void *const *k_caches,
                                const void *const *v_caches, const void *const *k_new,
                                const void *const *v_new, const int32_t *seq_lens,
                                int32_t top_k, int32_t *idx_buf, int32_t idx_valid,
                                void *const *outs, float *const *outs_f32, void *ws,
                                size_t ws_bytes, void *stream, void *const *layer_events);
td_status td_plan_create_append(td_plan **plan, const td_shape *shape, int32_t num_layers,
                                const int32_t *modes, const void *const *q,
                                const void *const *k_caches, const void *const *v_caches,
                                const void *const *k_new, const void *const *v_new,
                                const int32_t *seq_lens, int32_t top_k, int32_t *idx_buf,
                                int32_t idx_valid, void *const *outs, float *const *outs_f32,
                                void *ws, size_t ws_bytes);

/*
 * Measurement aid (not part of the decode step): reads exactly the K/V rows
 * one full layer (idx == NULL) or one sparse layer (idx = its index set)
 * reads, with the same split plan, launch shape and 16-byte row loads as the
 * register-streamed attention kernel, but no arithmetic beyond an XOR (which
 * lands in sink[0..sink_words), device, caller-owned).  Timing it gives the
 * memory-system floor of that layer's access pattern on the device.
 * Invalid or padding index entries are skipped.  Errors: TD_ERR_INVALID_ARG
 * for null or misaligned pointers, sink_words < 1 or (sparse) top_k outside
 * [1, max_seq_len]; TD_ERR_CUDA if the launch fails.
 */
td_status td_probe_layer_reads(const td_shape *shape, const void *k_cache, const void *v_cache,
                               const int32_t *seq_lens, const int32_t *idx, int32_t top_k,
                               uint32_t *sink, int32_t sink_words, void *stream);

/*
 * Kernel tuning knobs (process-wide, not thread-safe; for sweeps):
 *   "full_ctas_per_sm", "sparse_ctas_per_sm": resident CTAs assumed per SM
 *          by the split plan (default: the occupancy of the kernel launched;
 *          register-streamed sparse kernels that fit 4 or more per SM are
 *          planned one below it, leaving room for the next layer's CTAs)
 *   "full_waves", "sparse_waves": target waves of CTAs per launch
 *   "host_copy": 1 (default) host-buffer plans created afterwards copy with
 *          kernels where the host buffers are mapped; 0 with the copy
 *          engines only (see td_plan_create_host); other values restore the
 *          default
 *   "sparse_splits": 1..256 splits per (batch, KV head) of sparse launches
 *          (then kept within "max_splits", at most one per 64 entries, and
 *          at least one per 2048 entries, the most a sparse CTA stages);
 *          other values restore the default (from the CTAs per SM and the
 *          waves)
 *   "max_splits": upper bound on splits per (batch, KV head)
 *   "cluster": 1 merges a (batch, KV head)'s splits (when 2..8) through a
 *              thread-block cluster; 0 (default) through global partials
 *   "attn_carveout": preferred shared-memory carveout of the attention kernels
 *                    in percent (0..100; negative = driver default)
 *   "full_staged": 1 stages the K/V rows of full (and full+select) layers
 *                  through a ring of shared-memory stages filled by bulk
 *                  asynchronous copies; 0 streams them straight into
 *                  registers; negative restores the default (staged when
 *                  num_q_heads / num_kv_heads >= 4)
 *   "sparse_staged": 1 stages the gathered rows of sparse layers through a
 *                  per-thread cp.async ring in shared memory; 2 through TMA
 *                  row gathers (cp.async.bulk.tensor tile::gather4, four
 *                  rows per copy) into the same ring (a launch whose cache
 *                  rows B x Hkv x Nmax reach 2^31, or a cache not 16-byte
 *                  aligned, returns TD_ERR_UNSUPPORTED_SHAPE); 0 streams them
 *                  into registers; negative (default) takes 1 when every CTA
 *                  of the register-streamed plan would gather at most 64
 *                  rows, else 0.  Applies to the CUDA-core kernels (not to
 *                  G = 4, 8 on the tensor cores)
 *   "mma": 1 (and the default) runs grouped-query layers with G = 4 or 8 on
 *          the tensor cores (mma.sync over the group's heads); 0 on the CUDA
 *          cores (where "full_staged" / "sparse_staged" apply); negative
 *          restores the default
 *   "full_prefetch": 0..4 rounds ahead whose K/V lines each warp of a
 *          register-streamed full or full+select kernel prefetches into L2;
 *          negative restores the default (1 on the tensor cores, 0 on the
 *          CUDA cores)
 *   "topk_warp_max": top-k threshold bins of up to this many candidates are
 *          finished by one warp, larger ones by block-wide radix passes
 *          (default 256)
 *   "topk_threads": 1024 or 512 threads per top-k row (512: two CTAs per
 *                   SM); other values restore the default: 512 when the
 *                   rows exceed one wave of 1024-thread CTAs (one per SM)
 *                   and nothing of the call follows the selection, or the
 *                   sparse layer that follows needs more than one wave of
 *                   CTAs; else 1024
 *   "topk_cluster": CTAs per row of a top-k selection: 1 (one CTA
 *          of "topk_threads"), or 2, 4, 8 (a thread-block cluster of
 *          1024-thread CTAs, each scanning a slice of the row, merged through
 *          distributed shared memory); other values restore the default
 *          (for rows of at least 32768 positions, the largest cluster for
 *          which rows x cluster fits one wave of SMs with at least 16384
 *          positions per CTA; else 1)
 *   "pdl", "topk_pdl": 0 turns off programmatic dependent launch between a
 *                   call's kernels / before the top-k kernel (default 1)
 *   "mma_full_tokens", "mma_sparse_tokens": tokens each warp of a
 *          tensor-core full (and full+select) / sparse kernel takes per round:
 *          8 (CTAs of 8 warps) or 16 (CTAs of 4 warps, both row groups of the
 *          MMA); 32 takes 16 per round with two rounds in flight per warp
 *          (the next round requested before this one's arithmetic); 64
 *          (sparse only) stages a CTA's rounds in a ring of two
 *          shared-memory buffers, one round in flight ahead of the one
 *          computed; defaults 16 for full layers and 64 for sparse layers;
 *          other values restore the default
 *   "early_trigger": rounds before the end of its last round at which a
 *          CTA (ring, register-streamed, cp.async-staged sparse and 16-token
 *          full kernels) lets the
 *          next kernel of the call launch; always after the CTA's own wait
 *          for the previous kernel (default 4; 0: after the last round;
 *          negative restores the default)
 *   "full_interleave": 1 (default) the splits of a (batch row, KV head) of a
 *          full layer take its 64-token rounds in turn (tensor cores with 16
 *          tokens per warp and one round in flight; CUDA cores register-
 *          streamed); 0 one contiguous chunk each; negative restores the
 *          default
 *   "wait_limit_us": microseconds after which a staged full-layer CTA stops
 *          waiting for a bulk copy (default 1 s).  A CTA that gives up waits
 *          (at the default limit) for every copy it issued, then joins the
 *          split merge with an empty partial and sets TD_FLAG_WAIT_TIMEOUT:
 *          the layer's output lacks that CTA's tokens and the workspace stays
 *          consistent for the next launch
 *   "wait_test": 1 makes the first stage wait of every staged full-layer CTA
 *          poll a barrier that nothing arrives on, so it runs out after
 *          "wait_limit_us" (tests of the failure report; no fault, no hang);
 *          0 (default) in normal use
 * Otherwise value <= 0 restores the default.  Unknown key -> TD_ERR_INVALID_ARG.
 */
td_status td_set_tuning(const char *key, int32_t value);

/* Number of splits per (batch, KV head) the next full (sparse = 0) or sparse
 * (sparse = 1) launch of this shape would use on the current device
 * (for byte accounting and tests). */
int32_t td_query_splits(const td_shape *shape, int32_t top_k, int32_t sparse);

/* Which attention kernel the next launch of this shape would run on the
 * current device with the current tuning: full (sparse = 0; top_k > 0 for a
 * full+select layer) or sparse (sparse = 1, top_k entries per index row).
 * Returns a static, NUL-terminated description (the kernel and how it gets
 * its K/V rows), or "invalid shape".  For reports and tests. */
const char *td_kernel_name(const td_shape *shape, int32_t top_k, int32_t sparse);

#ifdef __cplusplus
}
#endif

#endif /* TD_H_ */
