// unip_sched.cpp -- host-side construction of the packed and chunked batches
// that the attention, importance and selection calls consume.
//
// Two builders, both plain host C++ (no CUDA calls):
//
//  * Prepacking ("Prepacking: A Simple Method for Fast Prefilling and
//    Increased Throughput in Large Language Models", summary sections
//    "技术框架" and "关键设计"): prompts of different lengths are combined
//    with a bin-packing algorithm, and each prompt keeps its own positions
//    (restarting at 0) inside the packed stream.  The page does not name the
//    packing rule; this file uses first-fit decreasing: prompts longest first
//    (equal lengths by lower index), each placed in the lowest-numbered bin
//    with room, bins opened in order.
//
//  * Chunked prefill ("Chunked Prefill", Ultralytics glossary, section "Como
//    funciona o pre-preenchimento segmentado"): every step has a token
//    budget; each running decode contributes one token first, then chunks of
//    waiting prompts fill what is left; a prompt that does not fit continues
//    in the following steps, its KV cache growing chunk by chunk, until it is
//    complete and decoding begins.  Section "Tecnicas de servico
//    relacionadas": the cache lives in fixed-size pages (PagedAttention).
//
// First fit runs in O(n log n) with a max-tree over the bins' free room: the
// leftmost bin whose room is at least the prompt is found by one descent.
// Bins not yet opened hold the full capacity, so the descent opens the next
// bin by itself when no open bin has room.

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <vector>

#include "unip.h"
#include "unip_sched.h"

namespace {

// Leftmost leaf with value >= x in a max-tree over `n` leaves (all leaves
// start at `init`).  Returns the leaf index.
class FirstFitTree {
 public:
  FirstFitTree(int32_t n, int32_t init) {
    size_ = 1;
    while (size_ < n) size_ <<= 1;
    t_.assign(2 * static_cast<size_t>(size_), INT32_MIN);
    for (int32_t i = 0; i < n; ++i) t_[size_ + i] = init;
    for (int32_t i = size_ - 1; i >= 1; --i) t_[i] = std::max(t_[2 * i], t_[2 * i + 1]);
  }
  int32_t leftmost_at_least(int32_t x) const {
    if (t_[1] < x) return -1;
    int32_t i = 1;
    while (i < size_) i = (t_[2 * i] >= x) ? 2 * i : 2 * i + 1;
    return i - size_;
  }
  int32_t value(int32_t leaf) const { return t_[size_ + leaf]; }
  void set(int32_t leaf, int32_t v) {
    int32_t i = size_ + leaf;
    t_[i] = v;
    for (i >>= 1; i >= 1; i >>= 1) t_[i] = std::max(t_[2 * i], t_[2 * i + 1]);
  }

 private:
  int32_t size_;
  std::vector<int32_t> t_;
};

}  // namespace

extern "C" UNIP_API int32_t unip_ffd_pack(const int32_t *lengths, int32_t num_prompts, int32_t capacity,
                                          int32_t *order, int32_t *bin_cu, int32_t *num_bins) {
  if (num_prompts < 0 || capacity <= 0 || !num_bins) return UNIP_ERR_INVALID_ARGUMENT;
  if (num_prompts > 0 && (!lengths || !order || !bin_cu)) return UNIP_ERR_INVALID_ARGUMENT;
  if (num_prompts == 0) {
    if (bin_cu) bin_cu[0] = 0;
    *num_bins = 0;
    return UNIP_OK;
  }
  for (int32_t i = 0; i < num_prompts; ++i)
    if (lengths[i] < 0 || lengths[i] > capacity) return UNIP_ERR_INVALID_ARGUMENT;
  try {
    std::vector<int32_t> by_len(num_prompts);
    for (int32_t i = 0; i < num_prompts; ++i) by_len[i] = i;
    std::stable_sort(by_len.begin(), by_len.end(),
                     [&](int32_t a, int32_t b) { return lengths[a] > lengths[b]; });
    // Every prompt fits an empty bin, so at most num_prompts bins are opened.
    FirstFitTree room(num_prompts, capacity);
    std::vector<int32_t> bin_of(num_prompts);
    std::vector<int32_t> bin_count(num_prompts, 0);
    int32_t opened = 0;
    for (int32_t i : by_len) {
      const int32_t b = room.leftmost_at_least(lengths[i]);
      room.set(b, room.value(b) - lengths[i]);
      bin_of[i] = b;
      ++bin_count[b];
      opened = std::max(opened, b + 1);
    }
    // Prompts of a bin are listed in the order they were placed (FFD order).
    bin_cu[0] = 0;
    for (int32_t b = 0; b < opened; ++b) bin_cu[b + 1] = bin_cu[b] + bin_count[b];
    std::vector<int32_t> fill(bin_cu, bin_cu + opened);
    for (int32_t i : by_len) order[fill[bin_of[i]]++] = i;
    *num_bins = opened;
  } catch (const std::bad_alloc &) {
    return UNIP_ERR_TOO_LARGE;
  }
  return UNIP_OK;
}

extern "C" UNIP_API int32_t unip_pack_metadata(const int32_t *lengths, int32_t num_prompts,
                                               const int32_t *order, int32_t *cu_seqlens,
                                               int32_t *positions, int32_t *src_index) {
  if (num_prompts < 0 || !cu_seqlens) return UNIP_ERR_INVALID_ARGUMENT;
  if (num_prompts > 0 && (!lengths || !order)) return UNIP_ERR_INVALID_ARGUMENT;
  int64_t total = 0;
  for (int32_t i = 0; i < num_prompts; ++i) {
    if (lengths[i] < 0) return UNIP_ERR_INVALID_ARGUMENT;
    total += lengths[i];
  }
  if (total > INT32_MAX) return UNIP_ERR_TOO_LARGE;
  if (total > 0 && !positions) return UNIP_ERR_INVALID_ARGUMENT;
  try {
    // Offsets of the prompts in their original concatenation; also checks
    // that `order` is a permutation.
    std::vector<int32_t> src_off(num_prompts + 1, 0);
    for (int32_t i = 0; i < num_prompts; ++i) src_off[i + 1] = src_off[i] + lengths[i];
    std::vector<uint8_t> seen(num_prompts, 0);
    for (int32_t s = 0; s < num_prompts; ++s) {
      const int32_t p = order[s];
      if (p < 0 || p >= num_prompts || seen[p]) return UNIP_ERR_INVALID_ARGUMENT;
      seen[p] = 1;
    }
    cu_seqlens[0] = 0;
    for (int32_t s = 0; s < num_prompts; ++s) {
      const int32_t p = order[s];
      const int32_t base = cu_seqlens[s];
      for (int32_t t = 0; t < lengths[p]; ++t) {
        positions[base + t] = t;
        if (src_index) src_index[base + t] = src_off[p] + t;
      }
      cu_seqlens[s + 1] = base + lengths[p];
    }
  } catch (const std::bad_alloc &) {
    return UNIP_ERR_TOO_LARGE;
  }
  return UNIP_OK;
}

// ---------------------------------------------------------------------------
// Token-budget step builder.

namespace {

struct Request {
  int32_t prompt_len;
  int32_t max_new_tokens;
  int32_t computed;   // tokens whose K/V are (or, once the step runs, will be) in the cache
  int32_t generated;  // tokens sampled so far
  std::vector<int32_t> pages;
};

}  // namespace

struct unip_step_builder {
  int32_t token_budget;
  int32_t page_size;
  int32_t num_pages;
  int32_t max_pages_per_seq;
  int32_t max_seqs;
  int32_t chunk_multiple;
  std::vector<int32_t> free_pages;  // stack; back() is taken first
  std::vector<Request> requests;    // indexed by request id
  std::deque<int32_t> active;       // unfinished request ids in arrival order
  std::vector<int32_t> release;     // ids finished by the last step; pages freed at the next one
  struct Seg {
    int32_t id, start, len;
    bool prefill;
  };
  std::vector<Seg> segs;            // the step being built (capacity max_seqs)
};

extern "C" UNIP_API int32_t unip_step_builder_create(int32_t token_budget, int32_t page_size, int32_t num_pages,
                                                     int32_t max_pages_per_seq, int32_t max_seqs,
                                                     int32_t chunk_multiple, unip_step_builder **out) {
  if (!out) return UNIP_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  // A chunk that stops short of its prompt ends on a multiple of chunk_multiple; with a multiple
  // above the budget no such chunk fits and a prompt longer than the budget would never start.
  if (token_budget <= 0 || page_size <= 0 || num_pages < 0 || max_pages_per_seq <= 0 || max_seqs <= 0 ||
      chunk_multiple <= 0 || chunk_multiple > token_budget)
    return UNIP_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(max_pages_per_seq) * page_size > INT32_MAX ||
      static_cast<int64_t>(num_pages) * page_size > INT32_MAX)
    return UNIP_ERR_TOO_LARGE;
  unip_step_builder *sb = new (std::nothrow) unip_step_builder();
  if (!sb) return UNIP_ERR_TOO_LARGE;
  try {
    sb->token_budget = token_budget;
    sb->page_size = page_size;
    sb->num_pages = num_pages;
    sb->max_pages_per_seq = max_pages_per_seq;
    sb->max_seqs = max_seqs;
    sb->chunk_multiple = chunk_multiple;
    sb->free_pages.resize(num_pages);
    for (int32_t i = 0; i < num_pages; ++i) sb->free_pages[i] = num_pages - 1 - i;  // page 0 on top
    // A step never holds more than max_seqs segments or finishes more requests than that, and
    // freed pages never exceed the cache: with this room reserved, building a step allocates
    // nothing once it has started changing the state.
    sb->release.reserve(max_seqs);
    sb->segs.reserve(max_seqs);
  } catch (const std::bad_alloc &) {
    delete sb;
    return UNIP_ERR_TOO_LARGE;
  }
  *out = sb;
  return UNIP_OK;
}

extern "C" UNIP_API void unip_step_builder_destroy(unip_step_builder *sb) { delete sb; }

extern "C" UNIP_API int32_t unip_step_builder_add(unip_step_builder *sb, int32_t prompt_len,
                                                  int32_t max_new_tokens, int32_t *request_id) {
  if (!sb || prompt_len <= 0 || max_new_tokens <= 0) return UNIP_ERR_INVALID_ARGUMENT;
  // The last sampled token never enters the cache.
  const int64_t cached = static_cast<int64_t>(prompt_len) + max_new_tokens - 1;
  const int64_t pages = (cached + sb->page_size - 1) / sb->page_size;
  if (pages > sb->max_pages_per_seq || pages > sb->num_pages) return UNIP_ERR_TOO_LARGE;
  if (sb->requests.size() >= static_cast<size_t>(INT32_MAX)) return UNIP_ERR_TOO_LARGE;
  try {
    const int32_t id = static_cast<int32_t>(sb->requests.size());
    sb->requests.push_back(Request{prompt_len, max_new_tokens, 0, 0, {}});
    sb->requests.back().pages.reserve(static_cast<size_t>(pages));  // grows without allocating later
    sb->active.push_back(id);
    if (request_id) *request_id = id;
  } catch (const std::bad_alloc &) {
    return UNIP_ERR_TOO_LARGE;
  }
  return UNIP_OK;
}

extern "C" UNIP_API int32_t unip_step_builder_state(const unip_step_builder *sb, int32_t *prefilling,
                                                    int32_t *decoding, int32_t *free_pages) {
  if (!sb) return UNIP_ERR_INVALID_ARGUMENT;
  int32_t pre = 0, dec = 0;
  for (int32_t id : sb->active) {
    const Request &r = sb->requests[id];
    (r.computed < r.prompt_len ? pre : dec) += 1;
  }
  // Pages of requests finished by the last step count as free: the next
  // step returns them before it schedules anything.
  int64_t held = 0;
  for (int32_t id : sb->release) held += static_cast<int64_t>(sb->requests[id].pages.size());
  if (prefilling) *prefilling = pre;
  if (decoding) *decoding = dec;
  if (free_pages) *free_pages = static_cast<int32_t>(sb->free_pages.size() + held);
  return UNIP_OK;
}

extern "C" UNIP_API int32_t unip_step_builder_next(unip_step_builder *sb, const unip_step_buffers *buf,
                                                   unip_step_counts *counts) {
  if (!sb || !buf || !counts || !buf->cu_seqlens || !buf->positions || !buf->slot_mapping ||
      !buf->block_table || !buf->request_ids || !buf->seg_mask || !buf->finished_ids)
    return UNIP_ERR_INVALID_ARGUMENT;
  const int32_t ps = sb->page_size;

  // Pages of the requests the previous step finished go back on the stack,
  // last page first, so that a request's first page ends on top.
  for (int32_t id : sb->release) {
    std::vector<int32_t> &pg = sb->requests[id].pages;
    for (auto it = pg.rbegin(); it != pg.rend(); ++it) sb->free_pages.push_back(*it);
    std::vector<int32_t>().swap(pg);
  }
  sb->release.clear();

  using Seg = unip_step_builder::Seg;
  std::vector<Seg> &segs = sb->segs;
  segs.clear();
  int32_t budget_left = sb->token_budget;

  // Decodes first, one token each, in arrival order.  A decode whose token
  // starts a new page waits when no page is free.
  for (int32_t id : sb->active) {
    if (static_cast<int32_t>(segs.size()) == sb->max_seqs || budget_left == 0) break;
    Request &r = sb->requests[id];
    if (r.computed < r.prompt_len) continue;
    if (r.computed % ps == 0) {
      if (sb->free_pages.empty()) continue;
      r.pages.push_back(sb->free_pages.back());
      sb->free_pages.pop_back();
    }
    segs.push_back(Seg{id, r.computed, 1, false});
    --budget_left;
  }

  // Then prompt chunks, in arrival order, until the budget, the segment
  // limit or the free pages run out.  A chunk that does not finish its
  // prompt ends on a multiple of chunk_multiple (absolute positions).
  for (int32_t id : sb->active) {
    if (static_cast<int32_t>(segs.size()) == sb->max_seqs || budget_left == 0) break;
    Request &r = sb->requests[id];
    if (r.computed >= r.prompt_len) continue;
    const int32_t remaining = r.prompt_len - r.computed;
    const int64_t coverable =
        (static_cast<int64_t>(r.pages.size()) + static_cast<int64_t>(sb->free_pages.size())) * ps - r.computed;
    int64_t c = std::min<int64_t>({remaining, budget_left, coverable});
    if (c < remaining && sb->chunk_multiple > 1) {
      const int64_t end = (r.computed + c) / sb->chunk_multiple * sb->chunk_multiple;
      c = end - r.computed;
    }
    if (c <= 0) break;  // first come, first served: later prompts do not overtake
    const int32_t need = static_cast<int32_t>((r.computed + c + ps - 1) / ps);
    while (static_cast<int32_t>(r.pages.size()) < need) {
      r.pages.push_back(sb->free_pages.back());
      sb->free_pages.pop_back();
    }
    segs.push_back(Seg{id, r.computed, static_cast<int32_t>(c), true});
    budget_left -= static_cast<int32_t>(c);
  }

  // Emit the step and advance every scheduled request.
  int32_t n_tok = 0, n_dec = 0, n_fin = 0;
  const int32_t mp = sb->max_pages_per_seq;
  buf->cu_seqlens[0] = 0;
  for (size_t s = 0; s < segs.size(); ++s) {
    const Seg &g = segs[s];
    Request &r = sb->requests[g.id];
    for (int32_t t = 0; t < g.len; ++t) {
      const int32_t pos = g.start + t;
      buf->positions[n_tok + t] = pos;
      buf->slot_mapping[n_tok + t] = r.pages[pos / ps] * ps + pos % ps;
    }
    int32_t *row = buf->block_table + s * static_cast<size_t>(mp);
    const int32_t np = static_cast<int32_t>(r.pages.size());
    for (int32_t p = 0; p < mp; ++p) row[p] = p < np ? r.pages[p] : -1;
    buf->request_ids[s] = g.id;
    buf->seg_mask[s] = g.prefill ? 1 : 0;
    n_tok += g.len;
    buf->cu_seqlens[s + 1] = n_tok;
    n_dec += g.prefill ? 0 : 1;

    r.computed += g.len;
    bool done = false;
    if (g.prefill) {
      if (r.computed == r.prompt_len) {  // the step that completes the prompt samples the first token
        r.generated = 1;
        done = r.generated == r.max_new_tokens;
      }
    } else {
      r.generated += 1;
      done = r.generated == r.max_new_tokens;
    }
    if (done) {
      buf->finished_ids[n_fin++] = g.id;
      sb->release.push_back(g.id);
    }
  }
  if (n_fin > 0) {
    sb->active.erase(std::remove_if(sb->active.begin(), sb->active.end(),
                                    [&](int32_t id) {
                                      const Request &r = sb->requests[id];
                                      return r.computed >= r.prompt_len && r.generated == r.max_new_tokens;
                                    }),
                     sb->active.end());
  }
  counts->num_segs = static_cast<int32_t>(segs.size());
  counts->num_tokens = n_tok;
  counts->num_decode = n_dec;
  counts->num_finished = n_fin;
  return UNIP_OK;
}
