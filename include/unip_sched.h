/*
 * unip_sched.h -- host-side batch builders of libunip: the packed batch of
 * Prepacking and the token-budget step of chunked prefill.  They produce the
 * metadata that unip_prefill_attention, unip_block_importance and
 * unip_select_gather take (cu_seqlens, positions, block tables).
 *
 * Sources (page titles as given on the pages):
 *   [PP]  "Prepacking: A Simple Method for Fast Prefilling and Increased
 *         Throughput in Large Language Models" summary, sections "技术框架"
 *         and "关键设计": prompts are combined into compact bins by a
 *         bin-packing algorithm; positions restart for every prompt.
 *   [CP]  "Chunked Prefill" (Ultralytics glossary), section "Como funciona o
 *         pre-preenchimento segmentado": a per-step token budget; one token
 *         for each running decode first, then chunks of waiting prompts fill
 *         the rest; an unfinished prompt continues in later steps, its KV
 *         cache growing chunk by chunk, until it decodes.  Section "Tecnicas
 *         de servico relacionadas": the KV cache lives in fixed-size pages.
 *
 * Conventions
 *   - Every pointer here is HOST memory owned by the caller; nothing is
 *     launched on a GPU and no CUDA call is made.
 *   - Return value: UNIP_OK or a negative code of unip.h; on an error the
 *     outputs are unspecified and a step builder's state is unchanged.
 *   - A step builder is not thread-safe; one thread drives it.
 */
#ifndef UNIP_SCHED_H_
#define UNIP_SCHED_H_

#include <stdint.h>

#include "unip.h"

#ifdef __cplusplus
extern "C" {
#endif

/* [PP] First-fit-decreasing bin packing of prompt lengths.
 *   lengths     int32 [num_prompts], each in [0, capacity]
 *   capacity    tokens per bin (> 0)
 *   order       out int32 [num_prompts]: prompt indices in packed order, bin
 *               after bin; inside a bin in the order they were placed
 *   bin_cu      out int32 [num_prompts + 1]: bin b holds
 *               order[bin_cu[b] .. bin_cu[b+1]); entries past num_bins are
 *               left untouched
 *   num_bins    out
 * Rule: prompts are taken longest first (equal lengths: lower index first)
 * and each goes to the lowest-numbered bin whose free room is at least its
 * length, a new bin being opened when none has room.  The page names no
 * particular bin-packing rule; first-fit decreasing is the plain one.
 * Errors: INVALID_ARGUMENT for a NULL pointer, a negative count, capacity
 * <= 0 or a length outside [0, capacity]. */
UNIP_API int32_t unip_ffd_pack(const int32_t *lengths, int32_t num_prompts, int32_t capacity,
                               int32_t *order, int32_t *bin_cu, int32_t *num_bins);

/* [PP] Metadata of a packed stream that lists the prompts in `order`.
 *   lengths     int32 [num_prompts] (original prompt order)
 *   order       int32 [num_prompts]: a permutation of 0..num_prompts-1
 *   cu_seqlens  out int32 [num_prompts + 1]: segment s is prompt order[s]
 *   positions   out int32 [N]: restart at 0 for every prompt
 *   src_index   out int32 [N] or NULL: packed token i is token src_index[i]
 *               of the prompts concatenated in their original order (the
 *               row list that unip_gather_tokens takes to build the packed
 *               hidden states)
 * Errors: INVALID_ARGUMENT (NULL pointer, negative length, `order` not a
 * permutation), TOO_LARGE (N above INT32_MAX). */
UNIP_API int32_t unip_pack_metadata(const int32_t *lengths, int32_t num_prompts, const int32_t *order,
                                    int32_t *cu_seqlens, int32_t *positions, int32_t *src_index);

/* [CP] Token-budget step builder with a paged KV cache. */
typedef struct unip_step_builder unip_step_builder;

/* Outputs of one step, all caller-owned host arrays.  S = number of
 * segments of the step (<= max_seqs), N = its tokens (<= token_budget). */
typedef struct unip_step_buffers {
  int32_t *cu_seqlens;   /* [max_seqs + 1] */
  int32_t *positions;    /* [token_budget]: absolute positions; segment s's prefix is positions[cu_seqlens[s]] */
  int32_t *slot_mapping; /* [token_budget]: cache slot page * page_size + offset where token i's K/V belong */
  int32_t *block_table;  /* [max_seqs][max_pages_per_seq]: row s = the request's pages in logical order, -1 after */
  int32_t *request_ids;  /* [max_seqs] */
  uint8_t *seg_mask;     /* [max_seqs]: 1 = prompt chunk (scored by unip_block_importance), 0 = decode token */
  int32_t *finished_ids; /* [max_seqs]: requests whose last token this step samples */
} unip_step_buffers;

typedef struct unip_step_counts {
  int32_t num_segs;     /* S; 0 when nothing could be scheduled */
  int32_t num_tokens;   /* N */
  int32_t num_decode;   /* decode segments; they come first */
  int32_t num_finished; /* entries written to finished_ids */
} unip_step_counts;

/* Creates a builder.
 *   token_budget        tokens per step (> 0)
 *   page_size           tokens per KV page (> 0)
 *   num_pages           physical pages in the cache (>= 0)
 *   max_pages_per_seq   block-table width (> 0)
 *   max_seqs            most segments in one step (> 0)
 *   chunk_multiple      a chunk that does not finish its prompt ends on a
 *                       multiple of this absolute position (1 = any, at most
 *                       token_budget); with the selection block size here,
 *                       the blocks of every chunk line up with the prompt's
 *                       own blocks
 *   out                 out: the new builder (NULL on error)
 * Errors: INVALID_ARGUMENT for a value out of range, TOO_LARGE when page
 * counts overflow int32 slot numbers or memory runs out. */
UNIP_API int32_t unip_step_builder_create(int32_t token_budget, int32_t page_size, int32_t num_pages,
                                          int32_t max_pages_per_seq, int32_t max_seqs, int32_t chunk_multiple,
                                          unip_step_builder **out);

/* Frees a builder (NULL is allowed). */
UNIP_API void unip_step_builder_destroy(unip_step_builder *sb);

/* Queues a request: a prompt of prompt_len tokens (> 0) that will sample
 * max_new_tokens tokens (> 0).  Request ids are 0, 1, 2, ... in call order.
 * Its cache holds prompt_len + max_new_tokens - 1 tokens at the end (the last
 * sampled token is never fed back); TOO_LARGE when that needs more pages than
 * max_pages_per_seq or num_pages. */
UNIP_API int32_t unip_step_builder_add(unip_step_builder *sb, int32_t prompt_len, int32_t max_new_tokens,
                                       int32_t *request_id);

/* Builds the next step and advances the requests in it, assuming the step
 * will run.  Policy ([CP]):
 *   1. pages of the requests that the previous step finished are freed;
 *   2. every decoding request, in arrival order, adds one token at position
 *      = its cached length, while budget and max_seqs last; a decode whose
 *      token needs a new page and finds none free sits this step out;
 *   3. prompts with tokens left, in arrival order, add one chunk each:
 *      min(tokens left, budget left, tokens the free pages can hold), its end
 *      rounded down to a multiple of chunk_multiple unless it completes the
 *      prompt; the first prompt that gets no tokens ends the step (no
 *      overtaking).
 * The step that completes a prompt samples its first token; each decode
 * step samples one more; a request finishes when it has sampled
 * max_new_tokens.  Pages are taken from a stack of free pages, one page at a
 * time as a request's cache reaches it.  Nothing to schedule gives
 * num_segs = 0; if requests remain then (unip_step_builder_state), the
 * cache has no page for the next token of any of them and, as no request is
 * preempted, they stay blocked: num_pages must leave room for the requests
 * admitted.  Errors: INVALID_ARGUMENT for a NULL pointer. */
UNIP_API int32_t unip_step_builder_next(unip_step_builder *sb, const unip_step_buffers *buf,
                                        unip_step_counts *counts);

/* Requests with prompt tokens left, requests decoding, and free pages
 * (counting pages that the next step frees first).  Any output may be NULL. */
UNIP_API int32_t unip_step_builder_state(const unip_step_builder *sb, int32_t *prefilling, int32_t *decoding,
                                         int32_t *free_pages);

#ifdef __cplusplus
}
#endif

#endif /* UNIP_SCHED_H_ */
