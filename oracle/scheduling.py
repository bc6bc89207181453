"""Plain-Python oracle of the host batch builders -- TEST INFRASTRUCTURE.

Only the test suite may import this module.  It shares no code with the
library's host builders and restates the two policies step by step, with
lists and loops, for small inputs.

* Prepacking ("Prepacking: A Simple Method for Fast Prefilling and Increased
  Throughput in Large Language Models", summary sections "技术框架" and
  "关键设计"): prompts are combined into bins by bin packing and every prompt
  restarts its positions at 0.  The page does not say which bin-packing rule;
  the reading taken is first-fit decreasing (longest first, equal lengths by
  lower index; each prompt into the lowest-numbered open bin with room, else a
  new bin).

* Chunked prefill ("Chunked Prefill", Ultralytics glossary, section "Como
  funciona o pre-preenchimento segmentado"): each step has a token budget;
  running decodes get one token each first; waiting prompts then fill the
  rest in chunks; an unfinished prompt resumes in the next step until it is
  complete and starts decoding.  Readings where the page is silent: arrival
  order throughout; the first prompt that gets no tokens ends the step; a
  chunk that does not finish its prompt ends on a multiple of
  ``chunk_multiple``; the KV cache is paged (section "Tecnicas de servico
  relacionadas") and a decode whose token needs a page when none is free
  waits a step.  Which physical page a request gets is not fixed by the page,
  so this oracle tracks only how many pages are free; tests compare the
  library's page ids for validity, not for equality.
"""
from __future__ import annotations


def ffd_pack(lengths, capacity):
    """Bins as lists of prompt indices, in the order the prompts were placed."""
    idx = list(range(len(lengths)))
    # Longest first; Python's sort is stable, so equal lengths keep index order.
    idx.sort(key=lambda i: -lengths[i])
    bins = []   # [used, [prompt, ...]]
    for i in idx:
        if lengths[i] > capacity or lengths[i] < 0:
            raise ValueError("a prompt longer than the bin")
        placed = False
        for b in bins:
            if capacity - b[0] >= lengths[i]:
                b[0] += lengths[i]
                b[1].append(i)
                placed = True
                break
        if not placed:
            bins.append([lengths[i], [i]])
    return [b[1] for b in bins]


def ffd_order(lengths, capacity):
    """The packing of ffd_pack as (order, bin_cu): prompts in packed order and bin boundaries."""
    bins = ffd_pack(lengths, capacity)
    order = [i for b in bins for i in b]
    bin_cu = [0]
    for b in bins:
        bin_cu.append(bin_cu[-1] + len(b))
    return order, bin_cu


def pack_metadata(lengths, order):
    """cu_seqlens, positions (restarting per prompt) and source token indices."""
    starts = []
    acc = 0
    for n in lengths:
        starts.append(acc)
        acc += n
    cu = [0]
    pos = []
    src = []
    for p in order:
        for t in range(lengths[p]):
            pos.append(t)
            src.append(starts[p] + t)
        cu.append(cu[-1] + lengths[p])
    return cu, pos, src


class ChunkedScheduler:
    """The token-budget step policy, tracking free-page counts only."""

    def __init__(self, token_budget, page_size, num_pages, max_seqs, chunk_multiple=1):
        self.budget = token_budget
        self.page = page_size
        self.free = num_pages
        self.max_seqs = max_seqs
        self.mult = chunk_multiple
        self.reqs = []        # dicts: prompt, max_new, done (cached tokens), sampled, pages, finished
        self.to_free = []

    def add(self, prompt_len, max_new_tokens):
        self.reqs.append({"prompt": prompt_len, "max_new": max_new_tokens, "done": 0, "sampled": 0,
                          "pages": 0, "finished": False})
        return len(self.reqs) - 1

    def _pages_for(self, tokens):
        return -(-tokens // self.page)

    def step(self):
        """One step: list of (request, first position, length, is_prompt_chunk), finished ids."""
        for r in self.to_free:
            self.free += self.reqs[r]["pages"]
            self.reqs[r]["pages"] = 0
        self.to_free = []
        live = [i for i, r in enumerate(self.reqs) if not r["finished"]]
        segs = []
        left = self.budget
        # Decodes: one token each.
        for i in live:
            r = self.reqs[i]
            if len(segs) == self.max_seqs or left == 0:
                break
            if r["done"] < r["prompt"]:
                continue
            need = self._pages_for(r["done"] + 1) - r["pages"]
            if need > self.free:
                continue
            self.free -= need
            r["pages"] += need
            segs.append((i, r["done"], 1, False))
            left -= 1
        # Prompt chunks.
        for i in live:
            r = self.reqs[i]
            if len(segs) == self.max_seqs or left == 0:
                break
            if r["done"] >= r["prompt"]:
                continue
            rest = r["prompt"] - r["done"]
            fits_pages = (r["pages"] + self.free) * self.page - r["done"]
            c = min(rest, left, fits_pages)
            if c < rest and self.mult > 1:
                end = ((r["done"] + c) // self.mult) * self.mult
                c = end - r["done"]
            if c <= 0:
                break
            need = self._pages_for(r["done"] + c) - r["pages"]
            self.free -= need
            r["pages"] += need
            segs.append((i, r["done"], c, True))
            left -= c
        finished = []
        for (i, start, n, is_prompt) in segs:
            r = self.reqs[i]
            r["done"] += n
            if is_prompt:
                if r["done"] == r["prompt"]:
                    r["sampled"] = 1
            else:
                r["sampled"] += 1
            if r["done"] >= r["prompt"] and r["sampled"] == r["max_new"]:
                r["finished"] = True
                finished.append(i)
                self.to_free.append(i)
        return segs, finished
