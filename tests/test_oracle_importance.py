"""Pins for the oracle's block importance.

The reading pinned here (the review of UniPrefill, section 3, says only that
the sequence is cut into blocks whose importance is estimated at a
full-attention layer): the last min(B, n) query rows of a segment score its
own key blocks by the attention probability they put on each block, summed
over heads and normalised per segment.  Checks: exact rational closed form
for zero queries, a dominant key, normalisation, and the attention
probabilities recovered from torch SDPA with identity values.
"""
from fractions import Fraction

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from sparsified_long_context_gb300 import workloads as W


def _rand_bits(rng, shape):
    return W.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _imp(wl_q, wl_k, wl_v, cu, pos, hq, hkv, d, B, seg_mask=None, cache=None):
    kw = cache or {}
    _, lse = oracle.attention(wl_q, wl_k, wl_v, cu, pos, hq, hkv, d, **kw)
    return oracle.block_importance(wl_q, wl_k, lse, cu, hq, hkv, d, B, seg_mask=seg_mask)


def test_zero_query_closed_form_with_prefix_and_ragged_block():
    rng = np.random.default_rng(21)
    P, n, hq, hkv, d, B, page = 40, 53, 4, 2, 16, 16, 16
    q = np.zeros((n, hq, d), np.uint16)
    k_all, v_all = _rand_bits(rng, (P + n, hkv, d)), _rand_bits(rng, (P + n, hkv, d))
    n_pages = -(-P // page)
    perm = rng.permutation(n_pages).astype(np.int32)
    kc = np.zeros((n_pages, page, hkv, d), np.uint16)
    vc = np.zeros_like(kc)
    for p in range(n_pages):
        a, b = p * page, min(P, (p + 1) * page)
        kc[perm[p], : b - a], vc[perm[p], : b - a] = k_all[a:b], v_all[a:b]
    cu = np.array([0, n], np.int32)
    pos = np.arange(P, P + n, dtype=np.int32)
    imp, blk_cu = _imp(q, k_all[P:], v_all[P:], cu, pos, hq, hkv, d, B,
                       cache=dict(k_cache=kc, v_cache=vc, block_table=perm[None], page_size=page))
    nb = -(-n // B)
    assert list(blk_cu) == [0, nb]
    # q = 0: every visible key of row i (prefix included) has probability 1/(P+i+1)
    M = [Fraction(0)] * nb
    for i in range(n - B, n):
        for j in range(i + 1):
            M[j // B] += Fraction(hq, P + i + 1)
    tot = sum(M)
    expect = np.array([float(m / tot) for m in M])
    assert np.max(np.abs(imp - expect)) < 1e-13


def test_short_segment_window_is_whole_segment():
    # n < B: the window is all n rows and there is a single (ragged) block
    rng = np.random.default_rng(22)
    n, hq, hkv, d = 9, 2, 1, 16
    q, k, v = _rand_bits(rng, (n, hq, d)), _rand_bits(rng, (n, hkv, d)), _rand_bits(rng, (n, hkv, d))
    imp, blk_cu = _imp(q, k, v, np.array([0, n], np.int32), np.arange(n, dtype=np.int32), hq, hkv, d, 16)
    assert list(blk_cu) == [0, 1] and abs(imp[0] - 1.0) < 1e-15


def test_dominant_key_takes_its_block():
    n, hq, hkv, d, B = 96, 2, 1, 16, 16
    rng = np.random.default_rng(23)
    qf = np.zeros((n, hq, d), np.float32)
    kf = rng.standard_normal((n, hkv, d)).astype(np.float32)
    kf[:, :, 0] = 0.0
    jstar = 37                      # block 2
    kf[jstar, 0, :] = 0.0
    kf[jstar, 0, 0] = 16.0
    qf[n - B:, :, 0] = 16.0         # window rows: logit 16*16/4 = 64 on jstar, 0 elsewhere
    q, k = W.f32_to_bf16_bits(qf), W.f32_to_bf16_bits(kf)
    v = _rand_bits(rng, (n, hkv, d))
    imp, _ = _imp(q, k, v, np.array([0, n], np.int32), np.arange(n, dtype=np.int32), hq, hkv, d, B)
    assert imp[jstar // B] >= 1 - 1e-6


def test_each_scored_segment_sums_to_one_and_mask_skips_segments():
    wl = W.tiny_packed()
    mask = np.array([1, 0, 1, 1], np.uint8)
    imp, blk_cu = _imp(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, 4, 2, 64, 16, seg_mask=mask)
    assert list(np.diff(blk_cu)) == [3, 0, 4, 16]
    for s in range(4):
        a, b = blk_cu[s], blk_cu[s + 1]
        if b > a:
            assert abs(imp[a:b].sum() - 1.0) < 1e-12
            assert np.all(imp[a:b] >= 0)


def test_matches_probabilities_from_sdpa_identity_values():
    """Attention probabilities from torch SDPA (V = identity), summed over the window rows."""
    rng = np.random.default_rng(24)
    n, hq, hkv, d, B = 75, 4, 2, 32, 16
    q, k, v = _rand_bits(rng, (n, hq, d)), _rand_bits(rng, (n, hkv, d)), _rand_bits(rng, (n, hkv, d))
    imp, _ = _imp(q, k, v, np.array([0, n], np.int32), np.arange(n, dtype=np.int32), hq, hkv, d, B)
    qt = torch.from_numpy(W.bf16_bits_to_f32(q).astype(np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(W.bf16_bits_to_f32(k).astype(np.float64)).permute(1, 0, 2)[None]
    kt = kt.repeat_interleave(hq // hkv, dim=1)
    eye = torch.eye(n, dtype=torch.float64)[None, None].expand(1, hq, n, n)
    probs = F.scaled_dot_product_attention(qt, kt, eye, is_causal=True)[0]   # [hq, n, n]
    col = probs[:, n - B:, :].sum(dim=(0, 1)).numpy()                       # per key
    nb = -(-n // B)
    blocks = np.array([col[b * B:(b + 1) * B].sum() for b in range(nb)])
    assert np.max(np.abs(imp - blocks / blocks.sum())) < 1e-12
