"""Pins for the oracle's attention: library SDPA, the page's chunked demo, closed forms.

Each test checks the fp64 oracle against something that is not the oracle:
torch's scaled_dot_product_attention (the routine the "Chunked Prefill" page
uses), the chunked-equals-one-shot result printed on that page, the Prepacking
claim that packing changes only mask and positions, and closed forms.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from sparsified_long_context_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _rand_bits(rng, shape):
    return W.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _sdpa_causal(q, k, v, hq, hkv):
    """torch SDPA (fp64, CPU), one prompt, kv heads shared by contiguous query-head groups."""
    qt = torch.from_numpy(_f64(q)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(_f64(k)).permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    vt = torch.from_numpy(_f64(v)).permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("n,hq,hkv,d", [(1, 2, 1, 16), (57, 4, 2, 32), (130, 4, 4, 64), (200, 8, 2, 128)])
def test_single_prompt_matches_torch_sdpa(n, hq, hkv, d):
    rng = np.random.default_rng(100 + n)
    q, k, v = _rand_bits(rng, (n, hq, d)), _rand_bits(rng, (n, hkv, d)), _rand_bits(rng, (n, hkv, d))
    cu = np.array([0, n], np.int32)
    out, _ = oracle.attention(q, k, v, cu, np.arange(n, dtype=np.int32), hq, hkv, d)
    ref = _sdpa_causal(q, k, v, hq, hkv)
    assert np.max(np.abs(out - ref)) < 1e-12


def _paged(k_tokens, v_tokens, page_size, rng):
    """Scatter tokens into a shuffled page pool; returns (k_cache, v_cache, block_table row)."""
    n, hkv, d = k_tokens.shape
    n_pages = max(1, -(-n // page_size))
    perm = rng.permutation(n_pages + 3)[:n_pages].astype(np.int32)  # spare pages stay unused
    kc = np.zeros((n_pages + 3, page_size, hkv, d), np.uint16)
    vc = np.zeros_like(kc)
    for p in range(n_pages):
        a, b = p * page_size, min(n, (p + 1) * page_size)
        kc[perm[p], : b - a] = k_tokens[a:b]
        vc[perm[p], : b - a] = v_tokens[a:b]
    return kc, vc, perm


def _chunked_run(q, k, v, hq, hkv, d, chunk, page_size, rng):
    n = q.shape[0]
    outs, sizes = [], []
    for start in range(0, n, chunk):
        end = min(start + chunk, n)
        sizes.append(end - start)
        kw = {}
        if start > 0:
            kc, vc, perm = _paged(k[:start], v[:start], page_size, rng)
            kw = dict(k_cache=kc, v_cache=vc, block_table=perm[None, :], page_size=page_size)
        o, _ = oracle.attention(q[start:end], k[start:end], v[start:end], np.array([0, end - start], np.int32),
                                np.arange(start, end, dtype=np.int32), hq, hkv, d, **kw)
        outs.append(o)
    return np.concatenate(outs, axis=0), sizes


def test_chunked_equals_one_shot_page_demo():
    g = json.load(open(os.path.join(GOLDEN, "chunked_prefill_demo.json")))
    n, chunk, h, d = g["prompt_len"], g["chunk"], g["num_heads"], g["head_dim"]
    rng = np.random.default_rng(0)
    q, k, v = _rand_bits(rng, (n, h, d)), _rand_bits(rng, (n, h, d)), _rand_bits(rng, (n, h, d))
    full, _ = oracle.attention(q, k, v, np.array([0, n], np.int32), np.arange(n, dtype=np.int32), h, h, d)
    chunked, sizes = _chunked_run(q, k, v, h, h, d, chunk, 16, rng)
    assert len(sizes) == g["num_chunks"]
    assert sizes == g["chunk_sizes"]
    assert np.allclose(full, chunked, atol=g["allclose_atol"]) == g["allclose_result"]
    assert np.max(np.abs(full - chunked)) < 1e-12


def test_chunked_gqa_odd_chunks_and_pages():
    rng = np.random.default_rng(7)
    n, hq, hkv, d = 301, 4, 2, 32
    q, k, v = _rand_bits(rng, (n, hq, d)), _rand_bits(rng, (n, hkv, d)), _rand_bits(rng, (n, hkv, d))
    full = _sdpa_causal(q, k, v, hq, hkv)
    for chunk, page in [(100, 16), (37, 8), (128, 32)]:
        chunked, _ = _chunked_run(q, k, v, hq, hkv, d, chunk, page, rng)
        assert np.max(np.abs(full - chunked)) < 1e-12


def test_packed_equals_each_prompt_alone():
    wl = W.tiny_packed()
    hq, hkv, d = wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    out, lse = oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, hq, hkv, d)
    for s in range(wl.num_segs):
        a, b = wl.cu_seqlens[s], wl.cu_seqlens[s + 1]
        o1, l1 = oracle.attention(wl.q[a:b], wl.k[a:b], wl.v[a:b], np.array([0, b - a], np.int32),
                                  np.arange(b - a, dtype=np.int32), hq, hkv, d)
        assert np.array_equal(out[a:b], o1)
        assert np.array_equal(lse[a:b], l1)
        # and each prompt alone is plain causal SDPA
        assert np.max(np.abs(o1 - _sdpa_causal(wl.q[a:b], wl.k[a:b], wl.v[a:b], hq, hkv))) < 1e-12


def test_constant_keys_give_mean_of_visible_values_with_prefix():
    rng = np.random.default_rng(11)
    P, n, hq, hkv, d, page = 45, 70, 2, 1, 16, 16
    kvec = _rand_bits(rng, (1, hkv, d))
    k_all = np.repeat(kvec, P + n, axis=0)
    v_all = _rand_bits(rng, (P + n, hkv, d))
    q = _rand_bits(rng, (n, hq, d))
    kc, vc, perm = _paged(k_all[:P], v_all[:P], page, rng)
    out, lse = oracle.attention(q, k_all[P:], v_all[P:], np.array([0, n], np.int32),
                                np.arange(P, P + n, dtype=np.int32), hq, hkv, d,
                                k_cache=kc, v_cache=vc, block_table=perm[None], page_size=page)
    vf = _f64(v_all)[:, 0, :]
    counts = np.arange(P + 1, P + n + 1, dtype=np.float64)
    expect = np.cumsum(vf, axis=0)[P:] / counts[:, None]
    for h in range(hq):
        assert np.max(np.abs(out[:, h, :] - expect)) < 1e-12
    # every score equals s0 = q.k/sqrt(d); lse = s0 + ln(#visible)
    s0 = (_f64(q)[:, :, :] * _f64(kvec)[0, 0][None, None, :]).sum(-1) / math.sqrt(d)
    assert np.max(np.abs(lse - (s0 + np.log(counts)[:, None]))) < 1e-12


def test_zero_query_lse_is_log_count_and_single_token_is_v():
    rng = np.random.default_rng(12)
    lengths = [1, 5, 1, 33]
    n = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    pos = np.concatenate([np.arange(L) for L in lengths]).astype(np.int32)
    q = np.zeros((n, 2, 16), np.uint16)
    k, v = _rand_bits(rng, (n, 1, 16)), _rand_bits(rng, (n, 1, 16))
    out, lse = oracle.attention(q, k, v, cu, pos, 2, 1, 16)
    assert np.max(np.abs(lse - np.log(pos + 1.0)[:, None])) < 1e-13
    for s, L in enumerate(lengths):
        if L == 1:
            t = cu[s]
            assert np.array_equal(out[t, 0], _f64(v[t, 0]))
            assert np.array_equal(out[t, 1], _f64(v[t, 0]))


def test_page_permutation_leaves_output_bit_identical():
    rng = np.random.default_rng(13)
    P, n, hq, hkv, d = 100, 20, 4, 2, 32
    k_all, v_all = _rand_bits(rng, (P + n, hkv, d)), _rand_bits(rng, (P + n, hkv, d))
    q = _rand_bits(rng, (n, hq, d))
    res = []
    for _ in range(2):
        kc, vc, perm = _paged(k_all[:P], v_all[:P], 16, rng)
        o, l = oracle.attention(q, k_all[P:], v_all[P:], np.array([0, n], np.int32),
                                np.arange(P, P + n, dtype=np.int32), hq, hkv, d,
                                k_cache=kc, v_cache=vc, block_table=perm[None], page_size=16)
        res.append((o, l))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])


def test_rows_subset_matches_full():
    wl = W.tiny_packed()
    rows = np.array([0, 36, 37, 200, 455], np.int32)
    full, lf = oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, 4, 2, 64)
    part, lp = oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, 4, 2, 64, rows=rows)
    assert np.array_equal(full[rows], part) and np.array_equal(lf[rows], lp)


def test_rejects_non_contiguous_positions_and_missing_pages():
    wl = W.tiny_packed()
    bad = wl.positions.copy()
    bad[5] += 1
    with pytest.raises(oracle.OracleError):
        oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, bad, 4, 2, 64)
    pos = wl.positions.copy()
    pos[:37] += 16  # first segment now claims a 16-token prefix but no pages are given
    with pytest.raises(oracle.OracleError):
        oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, pos, 4, 2, 64)


def test_compacted_reduces_to_packed_when_nothing_was_dropped():
    """With every token kept, contiguous positions and the first position as prefix length, the
    compacted-stream oracle is the packed / chunked one, bit for bit."""
    wl = W.tiny_packed()
    pl = wl.positions[wl.cu_seqlens[:-1]]
    a = oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, 4, 2, 64)
    b = oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, 4, 2, 64, prefix_lens=pl)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    rng = np.random.default_rng(31)
    P, n, hq, hkv, d = 70, 45, 4, 2, 32
    k_all, v_all = _rand_bits(rng, (P + n, hkv, d)), _rand_bits(rng, (P + n, hkv, d))
    q = _rand_bits(rng, (n, hq, d))
    kc, vc, perm = _paged(k_all[:P], v_all[:P], 16, rng)
    kw = dict(k_cache=kc, v_cache=vc, block_table=perm[None], page_size=16)
    pos = np.arange(P, P + n, dtype=np.int32)
    a = oracle.attention(q, k_all[P:], v_all[P:], np.array([0, n], np.int32), pos, hq, hkv, d, **kw)
    b = oracle.attention(q, k_all[P:], v_all[P:], np.array([0, n], np.int32), pos, hq, hkv, d,
                         prefix_lens=np.array([P], np.int32), **kw)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_compacted_matches_sdpa_with_position_mask():
    """Kept tokens with gaps in their positions behind a cached prefix of a different length: torch SDPA
    over [prefix keys, own keys] with the mask 'prefix: always; own key u: pos[u] <= pos[t]'."""
    rng = np.random.default_rng(32)
    hq, hkv, d, page = 4, 2, 32, 16
    lengths, prefixes = [23, 1, 40], [37, 5, 0]
    segs_q, segs_k, segs_v, pos, pages = [], [], [], [], []
    kc_all, vc_all, bt_rows = [], [], []
    n_pages_total = 0
    for L, P in zip(lengths, prefixes):
        segs_q.append(_rand_bits(rng, (L, hq, d)))
        segs_k.append(_rand_bits(rng, (L, hkv, d)))
        segs_v.append(_rand_bits(rng, (L, hkv, d)))
        gaps = rng.integers(1, 4, L)                         # strictly increasing, with gaps
        pos.append((P + 3 + np.cumsum(gaps)).astype(np.int32))
        pk, pv = _rand_bits(rng, (P, hkv, d)), _rand_bits(rng, (P, hkv, d))
        npg = max(1, -(-P // page))
        kcs = np.zeros((npg, page, hkv, d), np.uint16)
        vcs = np.zeros_like(kcs)
        for p_ in range(npg):
            a_, b_ = p_ * page, min(P, (p_ + 1) * page)
            kcs[p_, : b_ - a_], vcs[p_, : b_ - a_] = pk[a_:b_], pv[a_:b_]
        kc_all.append(kcs)
        vc_all.append(vcs)
        bt_rows.append(np.arange(n_pages_total, n_pages_total + npg))
        pages.append((pk, pv))
        n_pages_total += npg
    max_p = max(len(r) for r in bt_rows)
    bt = np.full((len(lengths), max_p), -1, np.int32)
    for s_, r in enumerate(bt_rows):
        bt[s_, : len(r)] = r
    q, k, v = np.concatenate(segs_q), np.concatenate(segs_k), np.concatenate(segs_v)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    positions = np.concatenate(pos)
    out, lse = oracle.attention(q, k, v, cu, positions, hq, hkv, d, k_cache=np.concatenate(kc_all),
                                v_cache=np.concatenate(vc_all), block_table=bt, page_size=page,
                                prefix_lens=np.array(prefixes, np.int32))
    grp = hq // hkv
    for s_, (L, P) in enumerate(zip(lengths, prefixes)):
        pk, pv = pages[s_]
        K = np.concatenate([pk, segs_k[s_]])                 # [P + L, hkv, d]
        V = np.concatenate([pv, segs_v[s_]])
        mask = np.ones((L, P + L), bool)
        mask[:, P:] = pos[s_][None, :] <= pos[s_][:, None]
        qt = torch.from_numpy(_f64(segs_q[s_])).permute(1, 0, 2)[None]
        kt = torch.from_numpy(_f64(K)).permute(1, 0, 2)[None].repeat_interleave(grp, dim=1)
        vt = torch.from_numpy(_f64(V)).permute(1, 0, 2)[None].repeat_interleave(grp, dim=1)
        ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask))[0].permute(1, 0, 2)
        assert np.max(np.abs(out[cu[s_]:cu[s_ + 1]] - ref.numpy())) < 1e-12


def test_compacted_rejects_non_increasing_positions():
    rng = np.random.default_rng(33)
    q, k, v = _rand_bits(rng, (6, 2, 16)), _rand_bits(rng, (6, 1, 16)), _rand_bits(rng, (6, 1, 16))
    cu = np.array([0, 6], np.int32)
    with pytest.raises(oracle.OracleError):
        oracle.attention(q, k, v, cu, np.array([0, 2, 2, 5, 6, 9], np.int32), 2, 1, 16,
                         prefix_lens=np.array([0], np.int32))
