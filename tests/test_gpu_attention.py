"""GPU parity of unip_prefill_attention (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from sparsified_long_context_gb300 import workloads as W

from gpu_harness import (assert_close, bf16_tensor_to_f64, library_ffd, oracle_attention_rows, sample_rows,
                         LSE_ABS)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run(wl: W.Workload):
    from sparsified_long_context_gb300 import binding as B
    from sparsified_long_context_gb300.pipeline import DeviceInputs, StepBuffers, run_attention
    B.unip_get_device_status(clear=True)
    di = DeviceInputs.from_workload(wl, "cuda", with_hidden=False)
    bufs = StepBuffers(di, block_size=wl.block_size or 64)
    run_attention(di, bufs)
    torch.cuda.synchronize()
    st = B.unip_get_device_status(clear=True)
    assert st == 0, B.describe_status(st)
    return bf16_tensor_to_f64(bufs.out), bufs.lse.cpu().numpy().astype(np.float64)


def _check(wl, rows=None):
    out, lse = _run(wl)
    ref_o, ref_l = oracle_attention_rows(wl, rows)
    sel = slice(None) if rows is None else rows
    e = assert_close(out[sel], ref_o, what=f"{wl.name} out")
    assert_close(lse.T[sel], ref_l, max_abs=LSE_ABS, mean_abs=LSE_ABS, what=f"{wl.name} lse")
    return e


def test_tiny_packed_full():
    _check(W.tiny_packed())


@pytest.mark.parametrize("lengths,hq,hkv,d", [
    ([1], 2, 1, 64), ([1, 1, 1], 4, 2, 128), ([127, 128, 129], 4, 4, 64), ([0, 300, 0, 5], 8, 2, 128),
    ([256, 1, 383], 2, 2, 128), ([1000], 8, 1, 64),
    # groups of 16 and 32 heads (8 and 4 tokens per tile), an even group that does not divide 128, an odd one
    ([1, 37, 200], 16, 1, 64), ([3, 40, 129], 32, 1, 128), ([5, 70, 131], 12, 2, 64), ([9, 130], 6, 2, 128)])
def test_packed_edge_shapes(lengths, hq, hkv, d):
    _check(W.packed(lengths, hq, hkv, d, seed=sum(lengths) + hq + d))


def _chunk_with_prefix(P, n, hq, hkv, d, page, seed):
    """One segment continuing a P-token prefix held in shuffled pages."""
    rng = np.random.default_rng(seed)
    tot = P + n
    k_all = W.f32_to_bf16_bits(rng.standard_normal((tot, hkv, d), dtype=np.float32))
    v_all = W.f32_to_bf16_bits(rng.standard_normal((tot, hkv, d), dtype=np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((n, hq, d), dtype=np.float32))
    n_pages = max(1, -(-P // page))
    perm = rng.permutation(n_pages + 2)[:n_pages].astype(np.int32)
    kp = np.zeros((n_pages + 2, page, hkv, d), np.uint16)
    vp = np.zeros_like(kp)
    for p in range(n_pages):
        a, b = p * page, min(P, (p + 1) * page)
        kp[perm[p], : b - a], vp[perm[p], : b - a] = k_all[a:b], v_all[a:b]
    cache = W.PagedCache(n_pages + 2, page, hkv, d, "array", kp, vp)
    return W.Workload(f"prefix{P}_n{n}_p{page}", hq, hkv, d, np.array([0, n], np.int32),
                      np.arange(P, P + n, dtype=np.int32), q, k_all[P:], v_all[P:], cache=cache,
                      block_table=perm[None, :])


@pytest.mark.parametrize("P,n,page,d", [(16, 10, 16, 64), (45, 70, 16, 128), (128, 128, 16, 128),
                                        (300, 1, 32, 128), (1000, 257, 64, 64), (4096, 130, 128, 128),
                                        (513, 512, 16, 128)])
def test_prefix_from_pages(P, n, page, d):
    _check(_chunk_with_prefix(P, n, 4, 2, d, page, seed=P + n))


def _batch_with_prefixes(Ps, ns, hq, hkv, d, page, seed):
    """Several segments, each continuing its own prefix; all prefixes share one shuffled page pool."""
    rng = np.random.default_rng(seed)
    pages = [max(0, -(-P // page)) for P in Ps]
    total = sum(pages)
    perm = rng.permutation(total + 3).astype(np.int32)
    kp = np.zeros((total + 3, page, hkv, d), np.uint16)
    vp = np.zeros_like(kp)
    bt = np.full((len(Ps), max(max(pages), 1)), -1, np.int32)
    qs, ks, vs = [], [], []
    off = 0
    for s, (P, n) in enumerate(zip(Ps, ns)):
        k_all = W.f32_to_bf16_bits(rng.standard_normal((P + n, hkv, d), dtype=np.float32))
        v_all = W.f32_to_bf16_bits(rng.standard_normal((P + n, hkv, d), dtype=np.float32))
        for p in range(pages[s]):
            a, b = p * page, min(P, (p + 1) * page)
            phys = perm[off + p]
            kp[phys, : b - a], vp[phys, : b - a] = k_all[a:b], v_all[a:b]
            bt[s, p] = phys
        off += pages[s]
        qs.append(W.f32_to_bf16_bits(rng.standard_normal((n, hq, d), dtype=np.float32)))
        ks.append(k_all[P:])
        vs.append(v_all[P:])
    cu = np.concatenate([[0], np.cumsum(ns)]).astype(np.int32)
    pos = np.concatenate([np.arange(P, P + n) for P, n in zip(Ps, ns)]).astype(np.int32)
    cache = W.PagedCache(total + 3, page, hkv, d, "array", kp, vp)
    return W.Workload(f"decode_batch_g{hq // hkv}", hq, hkv, d, cu, pos, np.concatenate(qs), np.concatenate(ks),
                      np.concatenate(vs), cache=cache, block_table=bt)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 1, 64), (4, 2, 128), (6, 2, 64)])
def test_decode_batch_with_prefixes(hq, hkv, d):
    """Decode tokens and short chunks behind cached prefixes, as in a continuous-batching step."""
    Ps = [1000, 17, 300, 2048, 5, 64, 129, 0]
    ns = [1, 1, 2, 5, 33, 65, 1, 3]
    _check(_batch_with_prefixes(Ps, ns, hq, hkv, d, 16, seed=hq * 100 + d))


@pytest.mark.parametrize("hq,hkv,page,d,seed", [(32, 8, 16, 128, 21), (16, 2, 64, 64, 22), (12, 2, 32, 128, 23)])
def test_many_segments_with_prefixes(hq, hkv, page, d, seed):
    """More work items than SMs, mixing one- and two-tile items and paged prefixes of every length,
    so that each persistent CTA walks many items (the ring, the Q buffers and O run on across them)."""
    rng = np.random.default_rng(seed)
    S = 260
    ns = rng.integers(1, 300, S).tolist()
    ns[::7] = [1] * len(ns[::7])                       # decode-like segments
    Ps = rng.integers(0, 1500, S).tolist()
    Ps[::5] = [0] * len(Ps[::5])                       # some segments without a prefix
    wl = _batch_with_prefixes(Ps, ns, hq, hkv, d, page, seed)
    _check(wl, sample_rows(wl, 300))


@pytest.mark.parametrize("make", [
    lambda: W.packed([0, 300, 0, 5], 8, 2, 128, seed=313),                 # (token, head) rows, G 4
    lambda: W.packed([1000], 8, 1, 64, seed=1073),                          # G 8
    lambda: W.packed([5, 70, 131], 12, 2, 64, seed=282),                    # even G 6 that does not divide 128
    lambda: _chunk_with_prefix(513, 512, 4, 2, 128, 16, seed=1025),         # chunk behind a paged prefix
    lambda: _batch_with_prefixes([1000, 17, 300, 2048, 5, 64, 129, 0], [1, 1, 2, 5, 33, 65, 1, 3],
                                 32, 8, 128, 16, seed=3328),                # decode tokens and short chunks
], ids=["g4", "g8", "g6", "chunk", "decode_batch"])
def test_paired_and_single_items_agree(make):
    """Two-tile and one-tile work items visit every row's keys in the same order, so the
    outputs are bit-identical; one of them is also checked against the oracle."""
    from sparsified_long_context_gb300 import binding as B
    wl = make()
    res = {}
    try:
        for mode in (B.UNIP_ATTN_SCHEDULE_PAIRED, B.UNIP_ATTN_SCHEDULE_SINGLE):
            B.unip_set_attention_schedule(mode)
            res[mode] = _run(wl)
    finally:
        B.unip_set_attention_schedule(B.UNIP_ATTN_SCHEDULE_AUTO)
    (o1, l1), (o2, l2) = res[B.UNIP_ATTN_SCHEDULE_PAIRED], res[B.UNIP_ATTN_SCHEDULE_SINGLE]
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ref_o, ref_l = oracle_attention_rows(wl, None)
    assert_close(o2, ref_o, what=f"{wl.name} out (one-tile items)")
    assert_close(l2.T, ref_l, max_abs=LSE_ABS, mean_abs=LSE_ABS, what=f"{wl.name} lse (one-tile items)")


def test_chunked_equals_one_shot():
    one, chunks = W.chunked()
    outs = []
    for wl in chunks:
        o, _ = _run(wl)
        outs.append(o)
    chunked = np.concatenate(outs, 0)
    full, _ = _run(one)
    # GPU chunked vs GPU one-shot on every element, then both against the oracle on sampled rows
    assert_close(chunked, full, what="chunked vs one-shot (GPU)")
    rows = sample_rows(one, 160)
    ref, _ = oracle.attention(one.q, one.k, one.v, one.cu_seqlens, one.positions, 32, 8, 128, rows=rows)
    assert_close(chunked[rows], ref, what="chunked vs oracle")
    assert_close(full[rows], ref, what="one-shot vs oracle")


def test_prepacked_sampled():
    wl = W.prepacked(library_ffd)
    _check(wl, sample_rows(wl, 400))


def test_long_single_sampled():
    """The 32768-token prompt: the last row of every 128-row query tile (it sees the most keys of
    its tile), the importance window (the last 64 rows) and the stratified sample."""
    wl = W.long_single(d_model=0)
    n = wl.num_tokens
    rows = np.union1d(sample_rows(wl, 48), np.arange(127, n, 128))
    rows = np.union1d(rows, np.arange(n - 64, n)).astype(np.int32)
    _check(wl, rows)


def test_mixed_step_sampled():
    wl = W.mixed_step(d_model=0)
    rows = sample_rows(wl, 96)
    # keep the decode rows in the sample modest: each reads up to 32k cached keys
    dec = rows[rows < 256][:8]
    rows = np.concatenate([dec, rows[rows >= 256]]).astype(np.int32)
    _check(wl, rows)


def _compact(wl, B, rng, drop=0.5):
    """Drop random B-token blocks of every segment (first and last kept), as a selection would; returns
    the kept stream (q, k, v rows, cu_seqlens_kept, original positions) and each segment's prefix length."""
    cu = wl.cu_seqlens
    keep_rows, lens = [], []
    for s in range(wl.num_segs):
        a, b = int(cu[s]), int(cu[s + 1])
        n = b - a
        nb = -(-n // B) if n else 0
        kb = rng.random(nb) >= drop
        if nb:
            kb[0] = kb[-1] = True
        rows = [a + i for i in range(n) if kb[i // B]]
        keep_rows += rows
        lens.append(len(rows))
    rows = np.array(keep_rows, np.int64)
    cu_k = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return (wl.q[rows], wl.k[rows], wl.v[rows], cu_k, wl.positions[rows].astype(np.int32),
            wl.prefix_lens.astype(np.int32))


def _check_compacted(wl, B, seed, drop=0.5):
    from sparsified_long_context_gb300 import binding as Bd
    rng = np.random.default_rng(seed)
    q, k, v, cu_k, pos_k, plen = _compact(wl, B, rng, drop)
    hq, hkv, d = wl.num_heads_q, wl.num_heads_kv, wl.head_dim
    kw_o, kw_g = {}, {}
    if wl.cache is not None:
        kc, vc = wl.cache.pages_numpy(np.arange(wl.cache.num_pages))
        kw_o = dict(k_cache=kc, v_cache=vc, block_table=wl.block_table, page_size=wl.cache.page_size)
        kct, vct = wl.cache.to_torch("cuda")
        kw_g = dict(k_cache=kct, v_cache=vct, block_table=torch.from_numpy(wl.block_table).cuda(),
                    page_size=wl.cache.page_size)
    n = int(cu_k[-1])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.empty((n, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, n), dtype=torch.float32, device="cuda")
    Bd.unip_get_device_status(clear=True)
    Bd.unip_compacted_attention(dev(q).view(torch.bfloat16), dev(k).view(torch.bfloat16), dev(v).view(torch.bfloat16),
                                dev(cu_k), dev(pos_k), dev(plen), out, lse, num_heads_q=hq, num_heads_kv=hkv,
                                head_dim=d, **kw_g)
    torch.cuda.synchronize()
    st = Bd.unip_get_device_status(clear=True)
    assert st == 0, Bd.describe_status(st)
    ref_o, ref_l = oracle.attention(q, k, v, cu_k, pos_k, hq, hkv, d, prefix_lens=plen, **kw_o)
    assert_close(bf16_tensor_to_f64(out), ref_o, what="compacted out")
    assert_close(lse.cpu().numpy().astype(np.float64).T, ref_l, max_abs=LSE_ABS, mean_abs=LSE_ABS,
                 what="compacted lse")


@pytest.mark.parametrize("lengths,hq,hkv,d,B", [([300, 37, 700, 129], 8, 2, 128, 16), ([1000, 5, 64], 32, 8, 128, 64),
                                                ([513, 77], 4, 4, 64, 32)])
def test_compacted_stream_packed(lengths, hq, hkv, d, B):
    """Attention of a later layer over the kept tokens (original positions with gaps), no cached prefix."""
    _check_compacted(W.packed(lengths, hq, hkv, d, seed=sum(lengths)), B, seed=len(lengths) + B)


@pytest.mark.parametrize("hq,hkv,d,page", [(32, 8, 128, 16), (8, 2, 64, 64)])
def test_compacted_stream_with_prefixes(hq, hkv, d, page):
    """Kept tokens of chunks behind cached prefixes (paged), including single decode-like tokens."""
    wl = _batch_with_prefixes([1000, 17, 300, 2048, 0, 64], [200, 1, 130, 65, 300, 3], hq, hkv, d, page, seed=hq + d)
    _check_compacted(wl, 16, seed=page)
