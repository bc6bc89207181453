"""Property-based comparison of the library's host batch builders with the
oracle of oracle/scheduling.py over random budgets, page sizes, cache sizes,
chunk multiples and request mixes (no GPU)."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import scheduling as osch  # noqa: E402
from sparsified_long_context_gb300 import binding  # noqa: E402


@settings(max_examples=150, deadline=None)
@given(st.lists(st.integers(0, 300), min_size=0, max_size=60), st.integers(1, 300))
def test_ffd_pack_equals_oracle(lengths, extra):
    cap = max(lengths + [1]) + extra - 1
    order, bin_cu = binding.unip_ffd_pack(np.array(lengths, np.int32), cap)
    bins = [order[bin_cu[b]:bin_cu[b + 1]].tolist() for b in range(len(bin_cu) - 1)]
    assert bins == osch.ffd_pack(lengths, cap)


@st.composite
def scenarios(draw):
    budget = draw(st.integers(1, 64))
    page = draw(st.sampled_from([1, 2, 4, 8, 16]))
    mult = draw(st.sampled_from([m for m in (1, 2, 4, 8, 16) if m <= budget]))
    max_seqs = draw(st.integers(1, 8))
    reqs = draw(st.lists(st.tuples(st.integers(1, 90), st.integers(1, 6)), min_size=1, max_size=10))
    need = [-(-(L + m - 1) // page) for (L, m) in reqs]
    num_pages = draw(st.integers(max(need), sum(need) + 2))
    return budget, page, mult, max_seqs, reqs, need, num_pages


@settings(max_examples=120, deadline=None)
@given(scenarios())
def test_step_builder_equals_oracle(sc):
    budget, page, mult, max_seqs, reqs, need, num_pages = sc
    sb = binding.StepBuilder(budget, page, num_pages, max(need), max_seqs, mult)
    ref = osch.ChunkedScheduler(budget, page, num_pages, max_seqs, mult)
    for (L, m) in reqs:
        assert sb.add(L, m) == ref.add(L, m)
    held = {}
    for _ in range(5000):
        stp = sb.next()
        segs, fin = ref.step()
        cu = stp["cu_seqlens"]
        got = [[int(stp["request_ids"][s]), int(stp["positions"][cu[s]]), int(cu[s + 1] - cu[s]),
                int(stp["seg_mask"][s])] for s in range(len(cu) - 1)]
        assert got == [[i, a, n, int(p)] for (i, a, n, p) in segs]
        assert stp["finished_ids"].tolist() == fin
        for s, (i, a, n, _) in enumerate(segs):
            row = stp["block_table"][s]
            pages = row[row >= 0].tolist()
            assert len(pages) == -(-(a + n) // page)
            assert held.get(i, pages[:len(held.get(i, []))]) == pages[:len(held.get(i, []))]
            held[i] = pages
            pos = np.arange(a, a + n)
            assert np.array_equal(stp["slot_mapping"][cu[s]:cu[s + 1]], np.array(pages)[pos // page] * page + pos % page)
        live = [p for r, ps in held.items() if not ref.reqs[r]["finished"] or r in fin for p in ps]
        assert len(live) == len(set(live))                      # no page held by two requests
        for r in fin:
            held.pop(r, None)
        if not segs:
            break
    pre, dec, free = sb.state()
    assert free == ref.free + sum(ref.reqs[r]["pages"] for r in ref.to_free)
