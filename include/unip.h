/*
 * unip.h -- C ABI of libunip: packed / chunked long-context prefill attention
 * with block-wise dynamic sparsification, for NVIDIA GB300 (sm_103a).
 *
 * The path, in call order:
 *   unip_prefill_attention  causal attention of a packed token stream whose
 *                           segments may continue a cached prefix held in KV
 *                           pages; writes the output and the row log-sum-exp.
 *   unip_block_importance   per-block importance of each selected segment,
 *                           from the last query rows and the stored row LSE.
 *   unip_topp_select        fewest blocks per segment whose cumulative
 *                           importance reaches p, plus the compaction indices.
 *   unip_gather_tokens      copies the kept tokens' hidden-state rows into a
 *                           compacted stream.
 *
 * Sources (page titles as given on the pages):
 *   [CP]  "Chunked Prefill" (Ultralytics glossary).  Section "Como funciona o
 *         pre-preenchimento segmentado": each chunk attends to the cached K/V
 *         of all earlier chunks plus its own tokens with a causal mask over
 *         absolute positions, giving the one-pass result; the page's example
 *         calls scaled_dot_product_attention (softmax scale 1/sqrt(D)).
 *         Section "Tecnicas de servico relacionadas": PagedAttention stores
 *         the KV cache in fixed-size pages.
 *   [PP]  "Prepacking: A Simple Method for Fast Prefilling and Increased
 *         Throughput in Large Language Models" summary, sections "技术框架"
 *         and "关键设计": prompts of varying length are packed into one
 *         sequence; the attention mask and positional encoding are changed so
 *         that each prompt only sees itself (block-diagonal causal mask,
 *         positions restarting per prompt).
 *   [UP]  "[논문리뷰] UniPrefill: Universal Long-Context Prefill Acceleration
 *         via Block-wise Dynamic Sparsification" review.  Section 1 ("Top-p
 *         Token Selection"): the fewest blocks whose cumulative importance
 *         reaches a threshold p.  Section 3: the input is cut into blocks whose
 *         importance is estimated at a full-attention layer, and dropped
 *         tokens are left out of every later sub-layer.
 *
 * Conventions shared by every call
 *   - Every data pointer is DEVICE memory owned by the caller; the library
 *     never allocates, frees or keeps a pointer after the call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = legacy default stream) and never synchronise the host.
 *   - Layout is token-major: q [N][H_q][D], k and v [N][H_kv][D], bf16
 *     (passed as void*), rows contiguous.  Query head h reads kv head
 *     h / (H_q / H_kv) (contiguous groups).
 *   - Segment s holds tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 (int32,
 *     cu_seqlens[0] = 0, non-decreasing, cu_seqlens[S] = N).  Its positions
 *     must be contiguous; its cached-prefix length is positions[cu_seqlens[s]].
 *   - Return value: UNIP_OK, or a negative code for errors found on the host
 *     before any launch (nothing is enqueued then).  Errors that need the
 *     device's data (bad cu_seqlens, non-contiguous positions, bad page ids,
 *     a device wait that ran out) are recorded as bits of a per-device status
 *     word, read with unip_get_device_status; the affected call leaves its
 *     outputs unspecified.
 *   - A workspace buffer is not shared between calls that may overlap.
 */
#ifndef UNIP_H_
#define UNIP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define UNIP_API __attribute__((visibility("default")))

/* Host-side return codes. */
#define UNIP_OK 0
#define UNIP_ERR_INVALID_ARGUMENT (-1) /* null pointer, negative size, bad enum */
#define UNIP_ERR_UNSUPPORTED (-2)      /* shape the kernels do not cover */
#define UNIP_ERR_WORKSPACE (-3)        /* workspace missing, too small or misaligned */
#define UNIP_ERR_CUDA (-4)             /* CUDA runtime / launch failure */
#define UNIP_ERR_ALIGNMENT (-5)        /* pointer or row stride not 16-byte aligned */
#define UNIP_ERR_TOO_LARGE (-6)        /* beyond the noalloc scratch, a step builder's page budget, int32
                                          sizes or host memory */

/* Device status bits (unip_get_device_status). */
#define UNIP_DEV_BAD_SEQLENS 0x1u    /* cu_seqlens not monotone / ends wrong */
#define UNIP_DEV_BAD_POSITIONS 0x2u  /* positions not contiguous in a segment, or negative */
#define UNIP_DEV_BAD_PAGES 0x4u      /* prefix needs pages the block table does not give */
#define UNIP_DEV_TIMEOUT 0x8u        /* a bounded device wait ran out; kernel returned early */
#define UNIP_DEV_BAD_SCORES 0x10u    /* an importance score is negative, NaN or above 1 */
#define UNIP_DEV_TOO_MANY_BLOCKS 0x20u /* a segment has more blocks than Top-p supports */
#define UNIP_DEV_BAD_INDEX 0x40u     /* gather index out of range or n_kept above capacity */
#define UNIP_DEV_BAD_BLOCKS 0x80u    /* blk_cu does not match cu_seqlens and block_size */

/* Top-p flags. */
#define UNIP_KEEP_FIRST 0x1u /* always keep each segment's first block */
#define UNIP_KEEP_LAST 0x2u  /* always keep each segment's last block */

/* Largest number of blocks one segment may have in unip_topp_select. */
#define UNIP_TOPP_MAX_BLOCKS 8192

typedef struct unip_attn_params {
  int32_t num_heads_q;  /* H_q >= 1 */
  int32_t num_heads_kv; /* H_kv >= 1, divides H_q */
  int32_t head_dim;     /* D: 64 or 128 */
  float scale;          /* softmax scale; <= 0 selects 1/sqrt(D) */
} unip_attn_params;

/* Paged KV cache holding the cached prefixes ([CP], PagedAttention). */
typedef struct unip_paged_kv {
  const void *k_cache;          /* bf16 [num_pages][page_size][H_kv][D] */
  const void *v_cache;          /* bf16 [num_pages][page_size][H_kv][D] */
  int32_t num_pages;
  int32_t page_size;            /* tokens per page: 16, 32, 64 or 128 */
  const int32_t *block_table;   /* int32 [num_segs][max_pages_per_seq]; entry p of row s
                                   is the physical page of prefix tokens [p*page, (p+1)*page) */
  int32_t max_pages_per_seq;
} unip_paged_kv;

/* Library version string (static storage). */
UNIP_API const char *unip_version(void);

/* Text for a host return code (static storage). */
UNIP_API const char *unip_status_string(int32_t code);

/* Name of the last CUDA runtime error of the calling host thread (and clears
 * it): the detail behind a UNIP_ERR_CUDA return.  Static storage. */
UNIP_API const char *unip_last_cuda_error(void);

/* Reads the current device's status word into *bits (synchronises that
 * device), and clears it when clear != 0.  Returns UNIP_OK or UNIP_ERR_CUDA. */
UNIP_API int32_t unip_get_device_status(uint32_t *bits, int32_t clear);

/* Self-test of the bounded device waits (no page defines it; it checks the
 * library's error path).  Launches one CTA whose two roles wait on mbarriers
 * that nothing completes: the first gives up after limit_us microseconds
 * (1 .. 1000000) and raises UNIP_DEV_TIMEOUT; the second, waiting with the
 * kernels' own one-second limit, leaves as soon as it sees the first one's
 * abort.  gave_up: device int32 [3], receives {1, 1, microseconds the second
 * role waited}.  Nothing faults or hangs; the context stays usable.
 * Errors: INVALID_ARGUMENT (NULL gave_up, limit out of range). */
UNIP_API int32_t unip_selftest_bounded_wait(uint32_t limit_us, int32_t *gave_up, void *stream);

/* Shape of the attention work items, process-wide (all devices, all later
 * calls of unip_prefill_attention, unip_compacted_attention and the noalloc
 * variant).  A work item is two 128-row query tiles that share every K/V tile
 * (one tile's softmax overlaps the other's MMAs), or one tile.  AUTO takes one
 * tile per item when even twice the most two-tile items the call can hold
 * (from N, S and the heads) leave SMs idle -- a short chunk behind a long
 * prefix -- and two otherwise.  PAIRED and SINGLE force one shape (tests,
 * tuning); odd GQA groups always use one tile.  Results do not depend on the
 * shape beyond floating-point summation order, which is the same (every row's
 * keys are visited in the same tile order either way).
 * Errors: INVALID_ARGUMENT for an unknown mode. */
#define UNIP_ATTN_SCHEDULE_AUTO 0
#define UNIP_ATTN_SCHEDULE_PAIRED 1
#define UNIP_ATTN_SCHEDULE_SINGLE 2
UNIP_API int32_t unip_set_attention_schedule(int32_t mode);

/* ---------------------------------------------------------------------------
 * Attention ([CP] causal mask over absolute positions with a cached prefix,
 * [PP] block-diagonal mask and restarted positions).
 *
 * Token t of segment s (local index i, position P_s + i) with query head h
 * attends to the P_s prefix keys of its segment, read through block_table row
 * s, and to its segment's own tokens 0..i; nothing of other segments.
 *   out[t][h][:] = sum_j softmax_j(scale * q.k_j) v_j     (bf16, RNE)
 *   lse[h][t]    = ln sum_j exp(scale * q.k_j)            (fp32, may be NULL)
 * paged may be NULL when every segment starts at position 0.
 * Slots of a prefix's last page beyond the prefix must hold finite values.
 * workspace: device memory of unip_attention_workspace_size() bytes, 256-byte
 * aligned.  q, k, v, out, cache pointers: 16-byte aligned.
 * ------------------------------------------------------------------------- */
UNIP_API size_t unip_attention_workspace_size(int32_t total_tokens, int32_t num_segs,
                                              const unip_attn_params *prm);

/* The attention above over a packed / chunked stream.  Returns UNIP_OK, or a
 * host error code with nothing enqueued. */
UNIP_API int32_t unip_prefill_attention(const void *q, const void *k, const void *v,
                                        const int32_t *cu_seqlens, int32_t num_segs,
                                        const int32_t *positions, int32_t total_tokens,
                                        const unip_paged_kv *paged,
                                        const unip_attn_params *prm,
                                        void *out, float *lse,
                                        void *workspace, size_t workspace_bytes,
                                        void *stream);

/* ---------------------------------------------------------------------------
 * Attention over a compacted stream ([UP] section 3: the tokens a selection
 * dropped leave every later sub-layer): the kept tokens of each segment
 * (cu_seqlens_kept of unip_topp_select / unip_select_gather) with their
 * original positions, which increase inside a segment but may have gaps.
 * Token t of segment s attends to the prefix_lens[s] cached keys of its
 * segment (block_table row s; a later layer's cache holds kept tokens only,
 * so the prefix length is given, not derived from a position) and to its
 * segment's own tokens u with positions[u] <= positions[t]; nothing of other
 * segments.  prefix_lens: device int32 [num_segs], >= 0 (a bad value raises
 * UNIP_DEV_BAD_POSITIONS; non-increasing positions too).  Everything else,
 * including the workspace, as unip_prefill_attention.
 * ------------------------------------------------------------------------- */
UNIP_API int32_t unip_compacted_attention(const void *q, const void *k, const void *v,
                                          const int32_t *cu_seqlens, int32_t num_segs,
                                          const int32_t *positions, const int32_t *prefix_lens,
                                          int32_t total_tokens,
                                          const unip_paged_kv *paged,
                                          const unip_attn_params *prm,
                                          void *out, float *lse,
                                          void *workspace, size_t workspace_bytes,
                                          void *stream);

/* ---------------------------------------------------------------------------
 * Host-planned attention: the same operation as unip_prefill_attention /
 * unip_compacted_attention, with the work partition computed on the host.
 *
 * A serving step knows its batch layout on the host before anything runs
 * ([CP] "Como funciona o pre-preenchimento segmentado": the scheduler builds
 * each step from a token budget; unip_step_builder_next returns it).  From
 * host copies of cu_seqlens and of every segment's cached-prefix length the
 * plan cuts the call into work items, balances them over the SMs and passes
 * them to the kernel by value, so no planning kernel runs and no per-item
 * metadata is read from device memory.  One plan serves every attention call
 * of the step with that layout (every layer).
 *
 * A call with too few work items to fill the GPU (a short chunk behind a long
 * cached prefix, a few decode tokens with long contexts: [CP] "Ajustar o
 * orcamento de tokens", later chunks re-read the growing cache) also splits
 * the key range of its query tiles over several items; each item keeps fp32
 * partial results (unnormalised output, running maximum and sum) in the
 * workspace, and the last item of a tile to finish merges them in key order.
 * The merge order is fixed, so results do not depend on timing, but they
 * differ from the unsplit computation by floating-point rounding.
 *
 * unip_attention_plan_create
 *   cu_seqlens   host int32 [num_segs + 1] (cu[0] = 0, non-decreasing, cu[S] = total_tokens)
 *   prefix_lens  host int32 [num_segs]: cached keys before each segment's first token
 *                (the first position for a contiguous stream; the kept-prefix length for a
 *                compacted one); NULL: no segment has a prefix
 *   page_size, max_pages_per_seq: of the paged cache the calls will pass (ignored without prefixes)
 *   flags        UNIP_PLAN_NO_SPLIT: never split key ranges; UNIP_PLAN_SPLITS(n), 2 <= n <= 255:
 *                split every query unit's key range into min(n, its key tiles) items instead of
 *                letting the cost model decide (tuning, tests); UNIP_PLAN_DEVICE: use the device
 *                planner of unip_prefill_attention (as does any call the plan cannot hold:
 *                more than 128 segments or 1024 work items)
 *   num_sms      SMs of the device the calls will run on; 0: the current device's
 *   *plan        receives a host object; release it with unip_attention_plan_destroy.
 *   Errors: INVALID_ARGUMENT (bad sizes or metadata, a prefix longer than its pages, num_sms
 *   negative), UNSUPPORTED (head_dim, page size), TOO_LARGE (host memory).  Nothing touches
 *   the GPU except, with num_sms 0, a query of the current device's SM count.
 * unip_attention_plan_workspace_size: bytes of device workspace the runs need (256-aligned).
 * unip_attention_plan_info: info[0] 1 if host-planned, info[1] work items, info[2] CTAs,
 *   info[3] split query units, info[4] key splits in total, info[5] 1 if one query tile per item.
 * unip_prefill_attention_planned
 *   q, k, v, out, lse, paged: as unip_prefill_attention; q, k, v, out must hold the
 *   plan's total_tokens rows.  cu_seqlens, positions (and prefix_lens, NULL for a
 *   contiguous stream) are the device copies of the layout; only a device-planned
 *   plan reads them.  paged must match the plan's page size and max_pages_per_seq.
 *   workspace: >= unip_attention_plan_workspace_size bytes, 256-byte aligned, not
 *   shared with a call that may run at the same time.  The first run of a plan on a
 *   workspace clears the workspace's ticket area (one small memset on the stream).
 *   A plan may be used by one host thread at a time.
 * ------------------------------------------------------------------------- */
typedef struct unip_attn_plan unip_attn_plan;
#define UNIP_PLAN_NO_SPLIT 0x1
#define UNIP_PLAN_DEVICE 0x2
#define UNIP_PLAN_SPLITS(n) (((n) & 0xFF) << 8)
UNIP_API int32_t unip_attention_plan_create(const int32_t *cu_seqlens, int32_t num_segs,
                                            const int32_t *prefix_lens, int32_t total_tokens,
                                            const unip_attn_params *prm, int32_t page_size,
                                            int32_t max_pages_per_seq, int32_t flags, int32_t num_sms,
                                            unip_attn_plan **plan);
UNIP_API size_t unip_attention_plan_workspace_size(const unip_attn_plan *plan);
UNIP_API int32_t unip_attention_plan_info(const unip_attn_plan *plan, int32_t *info);
UNIP_API void unip_attention_plan_destroy(unip_attn_plan *plan);
UNIP_API int32_t unip_prefill_attention_planned(const unip_attn_plan *plan, const void *q, const void *k,
                                                const void *v, const int32_t *cu_seqlens,
                                                const int32_t *positions, const int32_t *prefix_lens,
                                                const unip_paged_kv *paged, void *out, float *lse,
                                                void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Attention without caller-provided workspace.  The paper has no counterpart:
 * this is a library convenience.  It computes exactly what
 * unip_prefill_attention computes, but its scratch (the tile plan) lives in a
 * fixed device array inside the library, so the call allocates nothing and
 * needs no workspace pointer.  It is meant for callers that cannot call
 * cudaMalloc or own a device allocator: a host that hands out only the
 * tensors it already owns (a plugin or custom-operator interface without an
 * allocator), or a latency-critical path that must not pay for an allocation
 * that may synchronise the device.
 *
 * Limit: ceil(total_tokens / 128) + num_segs <= UNIP_NOALLOC_MAX_TILES;
 * larger problems return UNIP_ERR_TOO_LARGE without enqueuing anything.
 * The array costs UNIP_NOALLOC_SCRATCH_BYTES of memory on every device that
 * loads the library, until the process exits.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture begins.
 * The address is kept for the life of the process: after cudaDeviceReset on
 * that device it is stale, and the entry point must not be called again.
 * Every call shares the one array per device: calls that may overlap on the
 * GPU (other streams, other host threads) race and must be serialised by the
 * caller.  Arguments, outputs and errors are those of unip_prefill_attention.
 * ------------------------------------------------------------------------- */
#define UNIP_NOALLOC_MAX_TILES 32768
#define UNIP_NOALLOC_SCRATCH_BYTES (256 + 8 * UNIP_NOALLOC_MAX_TILES)

UNIP_API int32_t unip_prefill_attention_noalloc(const void *q, const void *k, const void *v,
                                                const int32_t *cu_seqlens, int32_t num_segs,
                                                const int32_t *positions, int32_t total_tokens,
                                                const unip_paged_kv *paged,
                                                const unip_attn_params *prm,
                                                void *out, float *lse, void *stream);

/* ---------------------------------------------------------------------------
 * Block importance ([UP] section 3; scoring reading fixed by this library):
 * for each segment s with seg_mask[s] != 0 (all segments when seg_mask is
 * NULL) and n_s > 0 tokens, block b covers local tokens [b*B, min((b+1)*B, n_s)).
 * The last W = min(B, n_s) query rows score the segment's own keys:
 *   M_b = sum_{h < H_q} sum_{t in window} sum_{j in block b, j <= t}
 *         exp(scale * q_t^h . k_j - lse[h][t])
 *   imp_b = M_b / sum_b' M_b'.
 * lse is the row LSE written by unip_prefill_attention (prefix included).
 * Outputs: imp (fp32, capacity imp_capacity >= unip_importance_capacity()),
 * blk_cu (int32 [num_segs+1], block offsets; unscored segments own 0 blocks).
 * block_size: 16, 32, 64 or 128.
 * ------------------------------------------------------------------------- */
UNIP_API int32_t unip_importance_capacity(int32_t total_tokens, int32_t num_segs, int32_t block_size);

/* Bytes of device workspace unip_block_importance needs (work list and
 * per-kv-head partial masses); 0 for invalid arguments. */
UNIP_API size_t unip_importance_workspace_size(int32_t total_tokens, int32_t num_segs,
                                               int32_t block_size, const unip_attn_params *prm);

/* The importance above.  Returns UNIP_OK, or a host error code with nothing
 * enqueued; bad cu_seqlens raise UNIP_DEV_BAD_SEQLENS. */
UNIP_API int32_t unip_block_importance(const void *q, const void *k, const float *lse,
                                       const int32_t *cu_seqlens, int32_t num_segs,
                                       int32_t total_tokens, const uint8_t *seg_mask,
                                       int32_t block_size, const unip_attn_params *prm,
                                       float *imp, int32_t imp_capacity, int32_t *blk_cu,
                                       void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Top-p block selection ([UP] section 1) and compaction indices ([UP]
 * section 3).  Per segment with nb > 0 blocks, bit-exact and independent of
 * summation order:
 *   q_b = floor(imp_b * 2^32) (uint64), T = sum q_b, thr = p * (double)T;
 *   F = {first block if UNIP_KEEP_FIRST, last block if UNIP_KEEP_LAST};
 *   the other blocks ranked by imp descending, ties by lower index, are added
 *   in rank order while (double)(sum of kept q) < thr.  T == 0 keeps all.
 * Segments with zero blocks in blk_cu (not scored) keep every token.
 * Outputs: keep (uint8 per block), gather_idx (int32, kept source tokens in
 * original order, capacity total_tokens), cu_seqlens_kept (int32
 * [num_segs+1]), positions_kept (int32, original positions, capacity
 * total_tokens), n_kept (one int32, device).  0 <= p <= 1.
 * ------------------------------------------------------------------------- */
UNIP_API size_t unip_topp_workspace_size(int32_t total_tokens, int32_t num_segs, int32_t block_size);

/* The selection above.  Returns UNIP_OK, or a host error code with nothing
 * enqueued; invalid scores raise UNIP_DEV_BAD_SCORES. */
UNIP_API int32_t unip_topp_select(const float *imp, const int32_t *blk_cu,
                                  const int32_t *cu_seqlens, const int32_t *positions,
                                  int32_t num_segs, int32_t total_tokens, int32_t block_size,
                                  double p, uint32_t flags,
                                  uint8_t *keep, int32_t keep_capacity,
                                  int32_t *gather_idx, int32_t *cu_seqlens_kept,
                                  int32_t *positions_kept, int32_t *n_kept,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Top-p selection and compaction in one call ([UP] sections 1 and 3): the
 * outputs of unip_topp_select plus hidden_out[i][:] = hidden[gather_idx[i]][:]
 * (hidden: total_tokens rows with row stride row_stride; hidden_out: capacity
 * total_tokens rows with row stride out_row_stride; 16-byte aligned, d_model
 * and strides multiples of 8).  Same results as unip_topp_select followed by
 * unip_gather_tokens, with the index build folded into the gather so that the
 * call launches two kernels; the gather may start while Top-p finishes
 * (programmatic dependent launch).  With a single segment (num_segs == 1)
 * it is one launch: every CTA selects the segment's blocks itself and copies
 * its share of the kept rows.  Workspace as unip_topp_select.  With
 * hidden == hidden_out == NULL and d_model == 0 no rows are copied (the
 * selection and index outputs only).
 * ------------------------------------------------------------------------- */
UNIP_API int32_t unip_select_gather(const float *imp, const int32_t *blk_cu, const int32_t *cu_seqlens,
                                    const int32_t *positions, int32_t num_segs, int32_t total_tokens,
                                    int32_t block_size, double p, uint32_t flags,
                                    uint8_t *keep, int32_t keep_capacity,
                                    int32_t *gather_idx, int32_t *cu_seqlens_kept,
                                    int32_t *positions_kept, int32_t *n_kept,
                                    const void *hidden, int64_t row_stride, int32_t d_model,
                                    void *hidden_out, int64_t out_row_stride,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Importance, selection and compaction in one call ([UP] section 3: block
 * importance at a full-attention layer, then the Top-p block set of section
 * 1, then the dropped tokens leave the later sub-layers).  The outputs of
 * unip_block_importance (imp, blk_cu) and of unip_select_gather (keep,
 * gather_idx, cu_seqlens_kept, positions_kept, n_kept, hidden_out), with the
 * same bits: the normalisation and the selection of a segment run in one CTA
 * (the scores never make a round trip through memory before they are ranked),
 * and the row copy is a programmatic dependent of that grid.  Arguments as in
 * the two calls; workspace: unip_importance_select_gather_workspace_size()
 * bytes, 256-byte aligned.  Returns UNIP_OK or a host error code with nothing
 * enqueued; device errors as in the two calls.
 * ------------------------------------------------------------------------- */
UNIP_API size_t unip_importance_select_gather_workspace_size(int32_t total_tokens, int32_t num_segs,
                                                             int32_t block_size, const unip_attn_params *prm);
UNIP_API int32_t unip_importance_select_gather(
    const void *q, const void *k, const float *lse, const int32_t *cu_seqlens, const int32_t *positions,
    int32_t num_segs, int32_t total_tokens, const uint8_t *seg_mask, int32_t block_size,
    const unip_attn_params *prm, double p, uint32_t flags, float *imp, int32_t imp_capacity, int32_t *blk_cu,
    uint8_t *keep, int32_t *gather_idx, int32_t *cu_seqlens_kept, int32_t *positions_kept, int32_t *n_kept,
    const void *hidden, int64_t row_stride, int32_t d_model, void *hidden_out, int64_t out_row_stride,
    void *workspace, size_t workspace_bytes, void *stream);

/* Rotary position embedding of q and k in place, by each token's own
 * position, and append of the rotated k and of v into the paged KV cache.
 * [PP]: a packed stream restarts the positional encoding of every prompt,
 * so the positions passed here are the restarted ones (segment-local for
 * prompts without a prefix, absolute for chunks that continue one).  The
 * encoding is the rotary one (RoFormer): channel pair i of every head turns
 * by positions[t] * rope_theta^(-2i/D),
 *     (a, b) -> (a cos w - b sin w, b cos w + a sin w),
 * with pairs (i, i + D/2) when interleaved = 0 and (2i, 2i+1) when 1.  The
 * angle modulo one turn is exact integer arithmetic on a 64-bit fixed-point
 * turns-per-position value (double-precision frequency), so it stays within
 * ~1e-6 rad for any int32 position; the rotation is single precision and
 * the results are rounded to bf16 (RNE).
 * [CP]: a chunk's K/V join the paged cache that later chunks and decodes
 * attend to.
 *   q             bf16 [N][H_q][D], rotated in place; NULL skips q
 *   k             bf16 [N][H_kv][D], rotated in place
 *   v             bf16 [N][H_kv][D] (read only when appending)
 *   positions     int32 [N] (needed when rope_theta > 0)
 *   prm           H_q, H_kv, D (D a multiple of 16, 16..256); scale unused
 *   rope_theta    base of the frequencies (e.g. 10000 or 500000); <= 0
 *                 skips the rotation (append only)
 *   slot_mapping  int32 [N] or NULL (no append): token t's rotated k row and
 *                 v row go to slot s = page * page_size + offset of k_cache /
 *                 v_cache ([num_pages][page_size][H_kv][D] bf16); s < 0
 *                 skips the token (padding); s >= num_pages * page_size sets
 *                 UNIP_DEV_BAD_INDEX and skips it
 * Every pointer is 16-byte aligned device memory; asynchronous on `stream`.
 * Errors: INVALID_ARGUMENT (NULL where needed, negative sizes, interleaved
 * not 0/1, NaN or infinite theta), UNSUPPORTED (D), ALIGNMENT. */
UNIP_API int32_t unip_rope_append_kv(void *q, void *k, const void *v, const int32_t *positions, int32_t num_tokens,
                                     const unip_attn_params *prm, double rope_theta, int32_t interleaved,
                                     const int32_t *slot_mapping, void *k_cache, void *v_cache, int32_t num_pages,
                                     int32_t page_size, void *stream);

/* ---------------------------------------------------------------------------
 * Row gather ([UP] section 3: the kept tokens' hidden states form the stream
 * of the later layers):  out[i][:] = hidden[gather_idx[i]][:] for
 * i < *n_kept (read on the device), bit for bit.  hidden holds num_rows rows
 * of d_model bf16 values with row stride row_stride elements; out rows have
 * stride out_row_stride elements; capacity bounds *n_kept.  Pointers and
 * strides must be 16-byte aligned (d_model, strides multiples of 8).
 * ------------------------------------------------------------------------- */
UNIP_API int32_t unip_gather_tokens(const void *hidden, int32_t num_rows, int64_t row_stride,
                                    int32_t d_model, const int32_t *gather_idx,
                                    const int32_t *n_kept, int32_t capacity,
                                    void *out, int64_t out_row_stride, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* UNIP_H_ */
