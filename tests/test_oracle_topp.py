"""Pins for the oracle's Top-p block selection and compaction.

The review of UniPrefill (section 1, "Top-p token selection") defines the
selection as the fewest blocks whose cumulative importance reaches p.  The
brute force below enumerates every admissible subset on tiny inputs; the
special cases p = 0, p = 1 and zero mass follow from that definition.
"""
import itertools

import numpy as np
import pytest

import oracle
from sparsified_long_context_gb300 import workloads as W


def _q(imp):
    return np.floor(imp.astype(np.float64) * 2.0**32).astype(np.uint64)


def _forced(nb, flags):
    f = set()
    if flags & oracle.KEEP_FIRST:
        f.add(0)
    if flags & oracle.KEEP_LAST:
        f.add(nb - 1)
    return f


def _brute_min_count(imp, p, flags):
    nb = len(imp)
    qv = _q(imp)
    T = int(qv.sum())
    thr = p * float(T)
    F = _forced(nb, flags)
    rest = [b for b in range(nb) if b not in F]
    for extra in range(len(rest) + 1):
        for comb in itertools.combinations(rest, extra):
            mass = sum(int(qv[b]) for b in F) + sum(int(qv[b]) for b in comb)
            if float(mass) >= thr:
                return len(F) + extra
    return nb


def _random_imp(rng, nb, ties=False):
    x = rng.random(nb).astype(np.float64) ** 3
    if ties:
        x = np.round(x * 4) / 4 + 0.01
    x = (x / x.sum()).astype(np.float32)
    return x


@pytest.mark.parametrize("flags", [3, 1, 2, 0])
@pytest.mark.parametrize("ties", [False, True])
def test_bruteforce_minimal_and_tie_rule(flags, ties):
    rng = np.random.default_rng(31 + flags + 10 * ties)
    for trial in range(60):
        nb = int(rng.integers(1, 13))
        imp = _random_imp(rng, nb, ties)
        p = float(rng.choice([0.0, 0.3, 0.5, 0.8, 0.9, 0.95, 0.999, 1.0]))
        keep = oracle.topp_select(imp, np.array([0, nb], np.int32), p, flags)
        F = _forced(nb, flags)
        chosen = set(np.nonzero(keep)[0].tolist())
        assert F <= chosen
        assert len(chosen) == _brute_min_count(imp, p, flags)
        qv = _q(imp)
        assert float(sum(int(qv[b]) for b in chosen)) >= p * float(qv.sum()) or len(chosen) == nb
        # tie rule: every added block outranks every block left out
        bits = imp.view(np.uint32)
        added = [b for b in chosen if b not in F]
        left = [b for b in range(nb) if b not in chosen]
        for a in added:
            for l in left:
                assert bits[a] > bits[l] or (bits[a] == bits[l] and a < l)


def test_special_cases():
    rng = np.random.default_rng(40)
    imp = _random_imp(rng, 9)
    bc = np.array([0, 9], np.int32)
    assert set(np.nonzero(oracle.topp_select(imp, bc, 0.0))[0]) == {0, 8}
    imp2 = imp.copy()
    imp2[3] = 0.0
    imp2[5] = 0.0
    keep = oracle.topp_select(imp2, bc, 1.0)
    assert set(np.nonzero(keep)[0]) == {0, 8} | {b for b in range(9) if imp2[b] > 0}
    zero = np.zeros(5, np.float32)
    assert oracle.topp_select(zero, np.array([0, 5], np.int32), 0.5).tolist() == [1] * 5
    one = np.array([1.0], np.float32)
    assert oracle.topp_select(one, np.array([0, 1], np.int32), 0.9).tolist() == [1]


def test_equal_scores_prefer_lower_index():
    imp = np.full(8, 0.125, np.float32)
    keep = oracle.topp_select(imp, np.array([0, 8], np.int32), 0.5)
    # forced {0, 7} carry 0.25; two more needed, lowest indices 1 and 2
    assert np.nonzero(keep)[0].tolist() == [0, 1, 2, 7]


def test_segments_are_independent():
    rng = np.random.default_rng(41)
    parts = [_random_imp(rng, n) for n in (3, 7, 4, 16)]
    imp = np.concatenate(parts)
    bc = np.array([0, 3, 10, 14, 30], np.int32)
    keep = oracle.topp_select(imp, bc, 0.9)
    for s, part in enumerate(parts):
        alone = oracle.topp_select(part, np.array([0, len(part)], np.int32), 0.9)
        assert np.array_equal(keep[bc[s]:bc[s + 1]], alone)


def test_index_build_and_gather():
    rng = np.random.default_rng(42)
    lengths = [37, 1, 64, 0, 255, 20]
    n = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    pos = np.concatenate([np.arange(L) + 7 * s for s, L in enumerate(lengths)]).astype(np.int32)
    B = 16
    scored = [1, 1, 1, 1, 1, 0]
    nbs = [(-(-L // B) if sc and L > 0 else 0) for L, sc in zip(lengths, scored)]
    bc = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
    keep = (rng.random(bc[-1]) < 0.5).astype(np.uint8)
    gi, ck, pk, m = oracle.index_build(keep, bc, cu, pos, B)
    expect_count = 0
    for s, L in enumerate(lengths):
        if nbs[s] == 0:
            expect_count += L
        else:
            for b in range(nbs[s]):
                if keep[bc[s] + b]:
                    expect_count += min(B, L - b * B)
    assert m == expect_count == ck[-1]
    assert np.all(np.diff(gi) > 0)
    assert np.array_equal(pk, pos[gi])
    for s in range(len(lengths)):
        seg = gi[ck[s]:ck[s + 1]]
        assert np.all((seg >= cu[s]) & (seg < cu[s + 1]))
        if nbs[s] == 0:
            assert len(seg) == lengths[s]
    # brute force, token by token: exactly the tokens of kept blocks (every token of an unscored
    # segment), in stream order, and the kept offsets are the running counts per segment
    expect, counts = [], [0]
    for s, L in enumerate(lengths):
        for i in range(L):
            if nbs[s] == 0 or keep[bc[s] + i // B]:
                expect.append(int(cu[s]) + i)
        counts.append(len(expect))
    assert gi.tolist() == expect
    assert ck.tolist() == counts
    hidden = W.f32_to_bf16_bits(rng.standard_normal((n, 24), dtype=np.float32))
    out = oracle.gather(hidden, gi)
    assert np.array_equal(out, hidden[gi])


def test_negative_zero_is_the_zero_score():
    """A score of -0 is the zero score: no mass, and ranked with (not above) the +0 scores."""
    imp = np.array([0.25, 0.0, 0.3, 0.0, 0.0, 0.2, 0.25], np.float32)
    neg = imp.copy()
    neg[[1, 4]] = np.float32(-0.0)
    assert np.signbit(neg[1]) and np.signbit(neg[4])
    bc = np.array([0, 7], np.int32)
    for p in (0.0, 0.5, 0.8, 0.95, 1.0):
        for flags in (0, 1, 2, 3):
            assert np.array_equal(oracle.topp_select(neg, bc, p, flags), oracle.topp_select(imp, bc, p, flags))
    # with no forced blocks and p = 1 the zero scores are never needed
    assert oracle.topp_select(neg, bc, 1.0, 0).tolist() == [1, 0, 1, 0, 0, 1, 1]
