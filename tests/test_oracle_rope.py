"""Pins of the rotary-embedding oracle (oracle/rope.py): identities of plane
rotations, complex multiplication, hand-computed frequencies, the relative-
position property, and the relation between the two channel layouts."""
import numpy as np
import pytest

from oracle import rope as orope


def _x(seed, n=7, h=3, d=16):
    return np.random.default_rng(seed).standard_normal((n, h, d))


@pytest.mark.parametrize("interleaved", [False, True])
def test_position_zero_is_identity(interleaved):
    x = _x(0)
    assert np.array_equal(orope.rope(x, np.zeros(7, np.int64), 10000.0, interleaved), x)


def test_one_pair_is_complex_multiplication():
    """D = 2: one pair at frequency theta^0 = 1, so a token at position p is the
    complex number a + ib times e^{ip}."""
    x = _x(1, n=50, h=2, d=2)
    pos = np.arange(50) * 37 - 400
    z = (x[..., 0] + 1j * x[..., 1]) * np.exp(1j * pos)[:, None]
    for inter in (False, True):
        y = orope.rope(x, pos, 500000.0, inter)
        assert np.allclose(y[..., 0], z.real, rtol=0, atol=1e-12)
        assert np.allclose(y[..., 1], z.imag, rtol=0, atol=1e-12)


def test_hand_computed_frequencies():
    """D = 4, theta = 10000: frequencies 1 and 10000^(-1/2) = 1/100.  At position
    100 the second pair (channels 1 and 3 in the half layout) turns by 1 rad
    and the first by 100 rad."""
    assert np.allclose(orope.inv_frequencies(4, 10000.0), [1.0, 0.01], rtol=1e-15)
    x = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    y = orope.rope(x, np.array([100]), 10000.0, False)[0, 0]
    c1, s1 = np.cos(1.0), np.sin(1.0)
    assert np.allclose([y[1], y[3]], [2 * c1 - 4 * s1, 4 * c1 + 2 * s1], atol=1e-12)
    c0, s0 = np.cos(100.0), np.sin(100.0)
    assert np.allclose([y[0], y[2]], [1 * c0 - 3 * s0, 3 * c0 + 1 * s0], atol=1e-12)


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotations_compose_and_keep_pair_norms(interleaved):
    x = _x(2, d=32)
    a = np.random.default_rng(3).integers(-5000, 5000, 7)
    b = np.random.default_rng(4).integers(0, 70000, 7)
    once = orope.rope(x, a + b, 10000.0, interleaved)
    twice = orope.rope(orope.rope(x, a, 10000.0, interleaved), b, 10000.0, interleaved)
    assert np.allclose(once, twice, rtol=0, atol=1e-9)
    pairs = (lambda v: (v[..., 0::2], v[..., 1::2])) if interleaved else (lambda v: (v[..., :16], v[..., 16:]))
    p0, p1 = pairs(x)
    r0, r1 = pairs(once)
    assert np.allclose(p0 ** 2 + p1 ** 2, r0 ** 2 + r1 ** 2, rtol=1e-12, atol=0)


@pytest.mark.parametrize("interleaved", [False, True])
def test_scores_depend_on_relative_position_only(interleaved):
    """<R(m) q, R(n) k> = <R(m - n) q, k>: the score of a query and a key sees
    only their distance, which is why restarting positions per prompt leaves
    each prompt's attention as if it were alone."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    for m, n in [(0, 0), (5, 3), (1000, 17), (40000, 39990), (7, 12)]:
        lhs = np.sum(orope.rope(q, [m], 10000.0, interleaved) * orope.rope(k, [n], 10000.0, interleaved))
        rhs = np.sum(orope.rope(q, [m - n], 10000.0, interleaved) * k)
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


def test_layouts_differ_by_a_channel_permutation():
    x = _x(6, d=16)
    pos = np.arange(7) * 911
    perm = np.r_[0:16:2, 1:16:2]            # even channels first, then odd
    inv = np.argsort(perm)
    half = orope.rope(x[..., perm], pos, 10000.0, False)[..., inv]
    assert np.allclose(half, orope.rope(x, pos, 10000.0, True), rtol=0, atol=1e-12)


def test_append_writes_rows_at_their_slots():
    k_cache = np.full((4, 4, 2, 8), -1.0)
    v_cache = np.full((4, 4, 2, 8), -2.0)
    rows_k = np.arange(3 * 2 * 8, dtype=np.float64).reshape(3, 2, 8)
    rows_v = -rows_k
    orope.append_to_cache(k_cache, v_cache, rows_k, rows_v, np.array([13, -1, 2]))
    assert np.array_equal(k_cache[3, 1], rows_k[0]) and np.array_equal(v_cache[3, 1], rows_v[0])
    assert np.array_equal(k_cache[0, 2], rows_k[2]) and np.array_equal(v_cache[0, 2], rows_v[2])
    untouched = np.ones((4, 4), bool)
    untouched[3, 1] = untouched[0, 2] = False
    assert np.all(k_cache[untouched] == -1.0) and np.all(v_cache[untouched] == -2.0)


def test_bf16_decode_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x7F7F], np.uint16)
    assert orope.bf16_bits_to_f64(bits).tolist() == [1.0, -1.0, 0.0, 3.140625, 3.3895313892515355e38]
