"""Shared helpers of the GPU parity tests: device runs through the C ABI and
oracle runs on the same seeded inputs (sampled rows for the large shapes)."""
from __future__ import annotations

import numpy as np

import oracle
from sparsified_long_context_gb300 import workloads as W

# Tolerances for attention outputs and importance scores on bf16 inputs of unit scale.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 2e-3


def library_ffd(lengths, capacity):
    """The library's first-fit-decreasing packer (host C++ of libunip), as (order, bin_cu)."""
    from sparsified_long_context_gb300 import binding as B
    return B.unip_ffd_pack(lengths, capacity)


def bf16_tensor_to_f64(t) -> np.ndarray:
    import torch
    return t.detach().float().cpu().numpy().astype(np.float64)


def sample_rows(wl: W.Workload, budget: int, seed: int = 0) -> np.ndarray:
    """Deterministic stratified sample of token rows: segment edges, 128-row tile
    edges inside segments, plus evenly spaced rows up to ``budget``."""
    cu = wl.cu_seqlens
    picks = set()
    for s in range(wl.num_segs):
        a, b = int(cu[s]), int(cu[s + 1])
        if b <= a:
            continue
        for off in (0, 1, 126, 127, 128, 129, 255, 256):
            if a + off < b:
                picks.add(a + off)
        picks.add(b - 1)
        picks.add(max(a, b - 2))
    n = wl.num_tokens
    if len(picks) > budget // 2:
        rng = np.random.default_rng(seed)
        picks = set(rng.choice(sorted(picks), budget // 2, replace=False).tolist())
    step = max(1, n // max(1, budget - len(picks)))
    picks.update(range(step // 2, n, step))
    return np.array(sorted(picks), dtype=np.int32)


def compact_cache_for_rows(wl: W.Workload, rows: np.ndarray):
    """Oracle cache arguments restricted to the pages the sampled rows' segments read."""
    if wl.cache is None:
        return {}
    segs = sorted({int(np.searchsorted(wl.cu_seqlens, r, side="right") - 1) for r in rows})
    P = wl.prefix_lens
    need = []
    for s in segs:
        np_s = -(-int(P[s]) // wl.cache.page_size)
        need.extend(int(x) for x in wl.block_table[s, :np_s])
    uniq = np.array(sorted(set(need)), dtype=np.int64) if need else np.zeros(1, np.int64)
    remap = {int(p): i for i, p in enumerate(uniq)}
    bt = np.zeros_like(wl.block_table)
    for s in segs:
        np_s = -(-int(P[s]) // wl.cache.page_size)
        bt[s, :np_s] = [remap[int(x)] for x in wl.block_table[s, :np_s]]
    kc, vc = wl.cache.pages_numpy(uniq)
    return dict(k_cache=kc, v_cache=vc, block_table=bt, page_size=wl.cache.page_size)


def oracle_attention_rows(wl: W.Workload, rows=None):
    kw = compact_cache_for_rows(wl, rows if rows is not None else np.arange(wl.num_tokens))
    return oracle.attention(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.positions, wl.num_heads_q, wl.num_heads_kv,
                            wl.head_dim, rows=rows, **kw)


def assert_close(got: np.ndarray, ref: np.ndarray, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"{what}: mean abs err {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())
