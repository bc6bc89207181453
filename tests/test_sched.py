"""The library's host batch builders (include/unip_sched.h), called through the
C ABI, against the oracle of oracle/scheduling.py.  No GPU is needed: these
calls run on the host.

Packing results are unique under the first-fit-decreasing rule and compare
exactly.  For the step builder the segment structure (requests, positions,
chunk lengths, decode/prompt kind, finished requests) is unique and compares
exactly; which physical page a request receives is the library's choice, so
the pages are checked for validity instead: slots agree with the block table,
no page is held by two live requests, a request keeps its pages, and free
plus held pages add up to the cache."""
import numpy as np
import pytest

from oracle import scheduling as osch
from sparsified_long_context_gb300 import binding


@pytest.mark.parametrize("seed", range(10))
def test_ffd_pack_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    cap = int(rng.integers(1, 5000))
    n = int(rng.integers(0, 400))
    if seed % 3 == 0:
        lengths = rng.integers(0, cap + 1, n)
    elif seed % 3 == 1:
        lengths = rng.choice(np.unique([0, 1, cap // 4, cap // 3, cap // 2, cap]), n)   # many ties
    else:
        lengths = np.clip(np.round(np.exp(np.log(max(cap, 2) / 8) + rng.standard_normal(n))), 1, cap)
    lengths = lengths.astype(np.int32)
    order, bin_cu = binding.unip_ffd_pack(lengths, cap)
    bins = [order[bin_cu[b]:bin_cu[b + 1]].tolist() for b in range(len(bin_cu) - 1)]
    assert bins == osch.ffd_pack(lengths.tolist(), cap)


def test_ffd_pack_prepacking_scale():
    """A 64-prompt lognormal batch into 16384-token bins, as the packed workload uses."""
    rng = np.random.default_rng(3)
    z = rng.standard_normal(64)
    lengths = np.clip(np.round(np.exp(np.log(512.0) + z)), 32, 8192).astype(np.int32)
    order, bin_cu = binding.unip_ffd_pack(lengths, 16384)
    bins = [order[bin_cu[b]:bin_cu[b + 1]].tolist() for b in range(len(bin_cu) - 1)]
    assert bins == osch.ffd_pack(lengths.tolist(), 16384)


def test_ffd_pack_large_input_first_fit_property():
    """100k prompts (the tree search is O(n log n)); checks the first-fit
    property on the library's own output."""
    rng = np.random.default_rng(7)
    cap = 65536
    lengths = rng.integers(1, cap + 1, 100_000).astype(np.int32)
    order, bin_cu = binding.unip_ffd_pack(lengths, cap)
    assert np.array_equal(np.sort(order), np.arange(lengths.size))
    loads = np.add.reduceat(lengths[order].astype(np.int64), bin_cu[:-1])
    assert loads.max() <= cap
    # the smallest prompt of every bin did not fit the final room of any earlier bin
    smallest = np.minimum.reduceat(lengths[order], bin_cu[:-1])
    prefix_min_room = np.minimum.accumulate(cap - loads)
    assert np.all(smallest[1:] > prefix_min_room[:-1])


def test_ffd_pack_edges_and_errors():
    order, bin_cu = binding.unip_ffd_pack(np.zeros(0, np.int32), 16)
    assert order.size == 0 and bin_cu.tolist() == [0]
    order, bin_cu = binding.unip_ffd_pack([0, 0, 0], 16)
    assert order.tolist() == [0, 1, 2] and bin_cu.tolist() == [0, 3]
    with pytest.raises(binding.UnipError):
        binding.unip_ffd_pack([5, 17], 16)
    with pytest.raises(binding.UnipError):
        binding.unip_ffd_pack([5, -1], 16)
    with pytest.raises(binding.UnipError):
        binding.unip_ffd_pack([5], 0)


@pytest.mark.parametrize("seed", range(5))
def test_pack_metadata_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 50))
    lengths = rng.integers(0, 300, n).astype(np.int32)
    order = rng.permutation(n).astype(np.int32)
    cu, pos, src = binding.unip_pack_metadata(lengths, order)
    cu_o, pos_o, src_o = osch.pack_metadata(lengths.tolist(), order.tolist())
    assert cu.tolist() == cu_o and pos.tolist() == pos_o and src.tolist() == src_o


def test_pack_metadata_rejects_a_non_permutation():
    with pytest.raises(binding.UnipError):
        binding.unip_pack_metadata([3, 4, 5], [0, 0, 2])
    with pytest.raises(binding.UnipError):
        binding.unip_pack_metadata([3, 4, 5], [0, 3, 1])


def _drive(budget, page, num_pages, max_pages, max_seqs, mult, reqs, max_steps=100000):
    sb = binding.StepBuilder(budget, page, num_pages, max_pages, max_seqs, mult)
    ref = osch.ChunkedScheduler(budget, page, num_pages, max_seqs, mult)
    for (L, m) in reqs:
        assert sb.add(L, m) == ref.add(L, m)
    owner = {}          # physical page -> request
    pages_of = {}       # request -> list of pages (logical order)
    for _ in range(max_steps):
        st = sb.next()
        segs, fin = ref.step()
        cu = st["cu_seqlens"]
        got = [[int(st["request_ids"][s]), int(st["positions"][cu[s]]) if cu[s + 1] > cu[s] else -1,
                int(cu[s + 1] - cu[s]), int(st["seg_mask"][s])] for s in range(len(cu) - 1)]
        assert got == [[i, a, n, int(p)] for (i, a, n, p) in segs]
        assert st["finished_ids"].tolist() == fin
        assert st["num_decode"] == sum(1 for s in segs if not s[3])
        for s, (i, a, n, p) in enumerate(segs):
            assert st["positions"][cu[s]:cu[s + 1]].tolist() == list(range(a, a + n))
            row = st["block_table"][s]
            held = row[row >= 0].tolist()
            assert np.all(row[len(held):] == -1)
            assert len(held) == -(-(a + n) // page)                      # exactly the pages its cache needs
            assert held[:len(pages_of.get(i, []))] == pages_of.get(i, [])  # pages never move
            for pg in held:
                assert 0 <= pg < num_pages
                assert owner.get(pg, i) == i                              # not held by another request
                owner[pg] = i
            pages_of[i] = held
            slots = st["slot_mapping"][cu[s]:cu[s + 1]]
            pos = np.arange(a, a + n)
            assert np.array_equal(slots, np.array(held)[pos // page] * page + pos % page)
        for r in fin:
            for pg in pages_of.pop(r):
                del owner[pg]
        pre, dec, free = sb.state()
        assert free == num_pages - sum(len(v) for v in pages_of.values())
        assert free == ref.free + sum(ref.reqs[r]["pages"] for r in ref.to_free)
        if not segs:
            return sb, ref
    raise AssertionError("did not drain")


@pytest.mark.parametrize("seed", range(12))
def test_step_builder_matches_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    page = int(rng.choice([1, 2, 4, 16]))
    budget = int(rng.integers(1, 48))
    mult = int(rng.choice([m for m in (1, 2, 4, 8) if m <= budget]))
    max_seqs = int(rng.integers(1, 10))
    reqs = [(int(rng.integers(1, 80)), int(rng.integers(1, 7))) for _ in range(int(rng.integers(1, 16)))]
    need = [-(-(L + m - 1) // page) for (L, m) in reqs]
    # a roomy cache on even seeds, a cache that just fits the largest request on odd ones
    num_pages = sum(need) if seed % 2 == 0 else max(need) + int(rng.integers(0, 3))
    sb, ref = _drive(budget, page, num_pages, max(need), max_seqs, mult, reqs)
    pre, dec, free = sb.state()
    if seed % 2 == 0:           # with room for everything every request completes
        assert (pre, dec, free) == (0, 0, num_pages)
        assert all(r["finished"] for r in ref.reqs)


@pytest.mark.parametrize("k", range(3))
def test_step_builder_hand_worked_traces(k):
    import json
    import os
    tr = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "chunked_schedule_traces.json")))
    tr = tr["traces"][k]
    sb = binding.StepBuilder(tr["token_budget"], tr["page_size"], tr["num_pages"], 64, tr["max_seqs"],
                             tr["chunk_multiple"])
    for (L, m) in tr["requests"]:
        sb.add(L, m)
    for step in tr["steps"]:
        st = sb.next()
        cu = st["cu_seqlens"]
        segs = [[int(st["request_ids"][s]), int(st["positions"][cu[s]]), int(cu[s + 1] - cu[s]),
                 int(st["seg_mask"][s])] for s in range(len(cu) - 1)]
        assert segs == step["segs"]
        assert st["finished_ids"].tolist() == step["finished"]
        if "free_pages_after" in step:
            assert sb.state()[2] == step["free_pages_after"]


def test_step_builder_mixed_step_shape():
    """256 running decodes plus 4 long prompts under an 8192-token budget with
    64-token chunk alignment: the first mixed step holds the 256 decode tokens
    first, then prompt chunks filling the rest, each ending on a multiple of 64."""
    page = 16
    sb = binding.StepBuilder(8192, page, 1 << 20, 8192, 512, 64)
    rng = np.random.default_rng(5)
    ctx = rng.integers(1024, 32769, 256)
    for c in ctx:
        sb.add(int(c), 1000)
    # bring every short request into decoding (prefill them first); a request
    # that finishes its prompt early decodes in the following steps
    decoded = np.zeros(256, np.int64)
    while sb.state()[0] > 0:
        st = sb.next()
        decoded[st["request_ids"][: st["num_decode"]]] += 1
    for _ in range(4):
        sb.add(65536, 16)
    st = sb.next()
    cu = st["cu_seqlens"]
    assert st["num_decode"] == 256
    assert cu[-1] == 8192
    assert np.all(np.diff(cu)[:256] == 1)
    chunks = np.diff(cu)[256:]
    assert chunks.tolist() == [7936]                   # arrival order: the first prompt takes the rest
    assert st["seg_mask"].tolist() == [0] * 256 + [1]
    assert st["request_ids"][:256].tolist() == list(range(256))
    assert np.array_equal(st["positions"][:256], (ctx + decoded).astype(np.int32))
    assert st["positions"][256] == 0 and st["request_ids"][256] == 256


def test_step_builder_rejects_bad_arguments():
    with pytest.raises(binding.UnipError):
        binding.StepBuilder(0, 16, 10, 4, 4)
    with pytest.raises(binding.UnipError):
        binding.StepBuilder(8, 16, 10, 4, 4, 0)
    with pytest.raises(binding.UnipError):
        binding.StepBuilder(8, 16, 10, 4, 4, 16)            # no partial chunk could ever fit the budget
    sb = binding.StepBuilder(8, 16, 10, 4, 4)
    with pytest.raises(binding.UnipError):
        sb.add(0, 1)
    with pytest.raises(binding.UnipError):
        sb.add(64, 2)            # 65 cached tokens need 5 pages > 4 per request
    assert sb.add(64, 1) == 0
    with pytest.raises(binding.UnipError):
        binding.StepBuilder(8, 1 << 16, 1 << 16, 4, 4)     # slot numbers overflow int32
